// The C ABI (include/thinmx.h): host-side validation, then one launch on
// the caller's stream.  Nothing here allocates device memory or
// synchronises, except the diagnostic tt_device_error_read.
#include <cmath>
#include <map>
#include <mutex>

#include "thinmx.h"
#include "common.cuh"
#include "launch.h"
#include "layout.cuh"
#include "tensor_map.h"

namespace tt {

// The library's device error word (first asynchronous error wins).
static __device__ int32_t g_device_error = 0;

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_info_ok[kMaxDevices];
std::mutex g_info_mu;
}  // namespace

const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_info_mu);
  if (!g_info_ok[dev]) {
    DeviceInfo d;
    d.device = dev;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return nullptr;
    if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
      return nullptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    d.error_word = static_cast<int32_t*>(p);
    g_info[dev] = d;
    g_info_ok[dev] = true;
  }
  return &g_info[dev];
}

EncodeTiledFn tensor_map_encoder() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

cudaError_t ensure_dynamic_smem(const void* kern, int device, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> granted;
  std::lock_guard<std::mutex> lock(mu);
  int& g = granted[{kern, device}];
  if (g >= bytes) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) g = bytes;
  return e;
}

}  // namespace tt

namespace {

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline tt_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return TT_OK;
  (void)cudaGetLastError();  // clear a sticky launch error so later calls see their own
  return TT_ERR_CUDA;
}

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1;
constexpr int64_t kMaxK = 16384;
constexpr int64_t kTcMinBatch = 4;  // smallest m sent to the tensor-core path
constexpr int64_t kMoeMaxHidden = 8192;
static_assert(TT_MOE_STATIC_MAX_HIDDEN == tt::kMoeStaticMaxHidden,
              "header limit and scratch array size must agree");

// Programmatic dependent launch on the hot-path kernels.
constexpr bool kPdl = true;

}  // namespace

extern "C" {

const char* tt_status_str(int status) {
  switch (status) {
    case TT_OK: return "TT_OK";
    case TT_ERR_NULL: return "TT_ERR_NULL";
    case TT_ERR_SHAPE: return "TT_ERR_SHAPE";
    case TT_ERR_ALIGN: return "TT_ERR_ALIGN";
    case TT_ERR_NONFINITE: return "TT_ERR_NONFINITE";
    case TT_ERR_UNSUPPORTED: return "TT_ERR_UNSUPPORTED";
    case TT_ERR_CUDA: return "TT_ERR_CUDA";
    case TT_ERR_TIMEOUT: return "TT_ERR_TIMEOUT";
    case TT_ERR_SIZE: return "TT_ERR_SIZE";
    default: return "TT_ERR_UNKNOWN";
  }
}

int tt_version(void) { return 10000; }

tt_status tt_device_error_read(int32_t* out) {
  if (!out) return TT_ERR_NULL;
  const tt::DeviceInfo* di = tt::device_info();
  if (!di) return TT_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return from_cuda(cudaErrorUnknown);
  int32_t v = 0;
  if (cudaMemcpy(&v, di->error_word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return from_cuda(cudaErrorUnknown);
  const int32_t zero = 0;
  if (cudaMemcpy(di->error_word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return from_cuda(cudaErrorUnknown);
  *out = v;
  return TT_OK;
}

tt_status tt_quantize_mxfp4(const float* w, int64_t n, int64_t k, uint8_t* codes,
                            uint8_t* scales, int32_t* status_dev, void* stream) {
  if (n < 0 || k < 0 || k % 32 != 0 || n > kMaxRows) return TT_ERR_SHAPE;
  if (n == 0 || k == 0) return TT_OK;
  if (!w || !codes || !scales) return TT_ERR_NULL;
  if (!aligned(w, 16) || !aligned(codes, 16) || (status_dev && !aligned(status_dev, 4)))
    return TT_ERR_ALIGN;
  return from_cuda(tt::launch_quantize_mxfp4(w, n, k, codes, scales, status_dev,
                                             as_stream(stream)));
}

tt_status tt_mxfp4_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k,
                              float* out, void* stream) {
  if (n < 0 || k < 0 || k % 32 != 0 || n > kMaxRows) return TT_ERR_SHAPE;
  if (n == 0 || k == 0) return TT_OK;
  if (!codes || !scales || !out) return TT_ERR_NULL;
  if (!aligned(out, 8)) return TT_ERR_ALIGN;
  return from_cuda(tt::launch_dequantize_mxfp4(codes, scales, n, k, out, as_stream(stream)));
}

size_t tt_mxfp4_swiglu_packed_bytes(int64_t n, int64_t k) {
  if (n < 1 || k < 32 || k % 32 != 0 || k > kMaxK || n > kMaxRows) return 0;
  return size_t(n) * size_t(tt::SwigluRecord(int(k)).bytes);
}

tt_status tt_mxfp4_pack_swiglu(const uint8_t* gate_codes, const uint8_t* gate_scales,
                               const float* gate_postscale, const uint8_t* up_codes,
                               const uint8_t* up_scales, const float* up_postscale, int64_t n,
                               int64_t k, void* packed, size_t packed_bytes, void* stream) {
  if (n < 1 || k < 32 || k % 32 != 0 || k > kMaxK || n > kMaxRows) return TT_ERR_SHAPE;
  if (!gate_codes || !gate_scales || !up_codes || !up_scales || !packed) return TT_ERR_NULL;
  if (packed_bytes < tt_mxfp4_swiglu_packed_bytes(n, k)) return TT_ERR_SIZE;
  if (!aligned(packed, 16) || (gate_postscale && !aligned(gate_postscale, 4)) ||
      (up_postscale && !aligned(up_postscale, 4)))
    return TT_ERR_ALIGN;
  return from_cuda(tt::launch_pack_swiglu(gate_codes, gate_scales, gate_postscale, up_codes,
                                          up_scales, up_postscale, n, k,
                                          static_cast<uint8_t*>(packed), as_stream(stream)));
}

tt_status tt_mxfp4_swiglu_matvec(const void* packed, int64_t n, int64_t k,
                                 const uint16_t* x_bf16, int64_t m, uint16_t* h_bf16,
                                 void* stream) {
  if (n < 1 || k < 32 || k % 32 != 0 || k > kMaxK || n > kMaxRows) return TT_ERR_SHAPE;
  if (m < 1 || m > 64) return TT_ERR_SHAPE;
  if (!packed || !x_bf16 || !h_bf16) return TT_ERR_NULL;
  if (!aligned(packed, 16) || !aligned(x_bf16, 16) || !aligned(h_bf16, 2)) return TT_ERR_ALIGN;
  // m = 2..8: the tile kernel with its multiply-adds on mma.sync, where its
  // x registers hold K (k <= 5120).  m = 1 streams records on the CUDA-core
  // kernels.  Otherwise m >= 4 goes to the tcgen05 kernel where k allows
  // (k % 64 == 0 and the shared-memory plan fits), and m <= 8 falls back to
  // the CUDA-core kernels.
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  cudaError_t e = cudaErrorInvalidConfiguration;  // "nothing launched"
  if (m >= 2 && m <= 8)
    e = tt::launch_swiglu_mxfp4_mma(pk, int(n), int(k), x_bf16, int(m), h_bf16, as_stream(stream),
                                    kPdl);
  if (e == cudaErrorInvalidConfiguration && (m > 8 || (m >= kTcMinBatch && k % 64 == 0)))
    e = tt::launch_swiglu_mxfp4_tc(pk, int(n), int(k), x_bf16, int(m), h_bf16, as_stream(stream),
                                   kPdl);
  if (m <= 8 && e == cudaErrorInvalidConfiguration)
    e = tt::launch_swiglu_mxfp4_cc(pk, int(n), int(k), x_bf16, int(m), h_bf16, as_stream(stream),
                                   kPdl);
  if (e == cudaErrorInvalidConfiguration) return TT_ERR_UNSUPPORTED;
  return from_cuda(e);
}

tt_status tt_bf16_swiglu_matvec(const uint16_t* wg, const uint16_t* wu, int64_t n, int64_t k,
                                const uint16_t* x_bf16, int64_t m, uint16_t* h_bf16,
                                void* stream) {
  if (n < 1 || k < 8 || k % 8 != 0 || k > (int64_t(1) << 30) || n > kMaxRows) return TT_ERR_SHAPE;
  if (m < 1 || m > 8) return TT_ERR_SHAPE;
  if (!wg || !wu || !x_bf16 || !h_bf16) return TT_ERR_NULL;
  if (!aligned(wg, 16) || !aligned(wu, 16) || !aligned(x_bf16, 16) || !aligned(h_bf16, 2))
    return TT_ERR_ALIGN;
  return from_cuda(tt::launch_swiglu_bf16(wg, wu, int(n), int(k), x_bf16, int(m), h_bf16,
                                          as_stream(stream), kPdl));
}

tt_status tt_mxfp4_matvec(const uint8_t* codes, const uint8_t* scales, const float* postscale,
                          int64_t n, int64_t k, const uint16_t* x_bf16, int64_t m,
                          uint16_t* y_bf16, void* stream) {
  if (n < 1 || k < 32 || k % 32 != 0 || k > kMaxK || n > kMaxRows) return TT_ERR_SHAPE;
  if (m < 1 || m > 8) return TT_ERR_SHAPE;
  if (!codes || !scales || !x_bf16 || !y_bf16) return TT_ERR_NULL;
  if (!aligned(codes, 16) || (postscale && !aligned(postscale, 4)) || !aligned(x_bf16, 16) ||
      !aligned(y_bf16, 2))
    return TT_ERR_ALIGN;
  const cudaError_t e = tt::launch_mxfp4_rows(codes, scales, postscale, int(n), int(k), x_bf16,
                                              int(m), y_bf16, as_stream(stream), kPdl);
  if (e == cudaErrorInvalidConfiguration) return TT_ERR_UNSUPPORTED;
  return from_cuda(e);
}

tt_status tt_bf16_matvec(const uint16_t* w, int64_t n, int64_t k, const uint16_t* x_bf16,
                         int64_t m, uint16_t* y_bf16, void* stream) {
  if (n < 1 || k < 8 || k % 8 != 0 || k > (int64_t(1) << 30) || n > kMaxRows) return TT_ERR_SHAPE;
  if (m < 1 || m > 8) return TT_ERR_SHAPE;
  if (!w || !x_bf16 || !y_bf16) return TT_ERR_NULL;
  if (!aligned(w, 16) || !aligned(x_bf16, 16) || !aligned(y_bf16, 2)) return TT_ERR_ALIGN;
  return from_cuda(tt::launch_bf16_rows(w, int(n), int(k), x_bf16, int(m), y_bf16,
                                        as_stream(stream), kPdl));
}

size_t tt_mxfp4_rows_packed_bytes(int64_t n, int64_t k) {
  if (n < 1 || k < 32 || k % 32 != 0 || k > kMaxK || n > kMaxRows) return 0;
  return size_t(tt::ColSlices(n, int(k)).bytes);
}

tt_status tt_mxfp4_pack_rows(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k,
                             void* packed, size_t packed_bytes, void* stream) {
  if (n < 1 || k < 32 || k % 32 != 0 || k > kMaxK || n > kMaxRows) return TT_ERR_SHAPE;
  if (!codes || !scales || !packed) return TT_ERR_NULL;
  if (packed_bytes < tt_mxfp4_rows_packed_bytes(n, k)) return TT_ERR_SIZE;
  if (!aligned(packed, 16)) return TT_ERR_ALIGN;
  return from_cuda(tt::launch_pack_rows(codes, scales, n, k, static_cast<uint8_t*>(packed),
                                        as_stream(stream)));
}

size_t tt_moe_workspace_bytes(int64_t hidden, int64_t inter, int32_t n_experts, int32_t top_k) {
  if (hidden < 32 || hidden > kMoeMaxHidden || inter < 32 || n_experts < 1 || n_experts > 256 || top_k < 1 || top_k > 8 ||
      top_k > n_experts)
    return 0;
  return tt::moe_workspace_bytes(hidden, inter, n_experts, top_k);
}

tt_status tt_moe_mxfp4_topk_mlp(const uint16_t* x_bf16, int64_t hidden, int64_t inter,
                                const uint16_t* router_w_bf16, int32_t n_experts, int32_t top_k,
                                const void* const* gate_up_packed, const void* const* down_packed,
                                uint16_t* out_bf16, int32_t* out_idx, float* out_prob,
                                void* workspace, size_t workspace_bytes, void* stream) {
  if (hidden < 32 || hidden % 32 != 0 || hidden > kMoeMaxHidden) return TT_ERR_SHAPE;
  if (inter < 32 || inter % 32 != 0 || inter > 8192) return TT_ERR_SHAPE;
  if (n_experts < 1 || n_experts > 256 || top_k < 1 || top_k > 8 || top_k > n_experts)
    return TT_ERR_SHAPE;
  if (!x_bf16 || !router_w_bf16 || !gate_up_packed || !down_packed || !out_bf16 || !out_idx ||
      !out_prob || !workspace)
    return TT_ERR_NULL;
  if (workspace_bytes < tt_moe_workspace_bytes(hidden, inter, n_experts, top_k))
    return TT_ERR_SIZE;
  if (!aligned(x_bf16, 16) || !aligned(router_w_bf16, 16) || !aligned(gate_up_packed, 8) ||
      !aligned(down_packed, 8) || !aligned(out_bf16, 2) || !aligned(out_idx, 4) ||
      !aligned(out_prob, 4) || !aligned(workspace, 16))
    return TT_ERR_ALIGN;
  const cudaError_t e = tt::launch_moe(
      x_bf16, int(hidden), int(inter), router_w_bf16, int(n_experts), int(top_k),
      reinterpret_cast<const uint8_t* const*>(gate_up_packed),
      reinterpret_cast<const uint8_t* const*>(down_packed), out_bf16, out_idx, out_prob,
      workspace, as_stream(stream), kPdl);
  if (e == cudaErrorInvalidConfiguration) return TT_ERR_UNSUPPORTED;
  return from_cuda(e);
}

tt_status tt_moe_mxfp4_topk_mlp_static(const uint16_t* x_bf16, int64_t hidden, int64_t inter,
                                       const uint16_t* router_w_bf16, int32_t n_experts,
                                       int32_t top_k, const void* const* gate_up_packed,
                                       const void* const* down_packed, uint16_t* out_bf16,
                                       int32_t* out_idx, float* out_prob, void* stream) {
  if (hidden < 32 || hidden % 32 != 0 || hidden > kMoeMaxHidden) return TT_ERR_SHAPE;
  if (inter < 32 || inter % 32 != 0 || inter > 8192) return TT_ERR_SHAPE;
  if (n_experts < 1 || n_experts > 256 || top_k < 1 || top_k > 8 || top_k > n_experts)
    return TT_ERR_SHAPE;
  if (hidden > TT_MOE_STATIC_MAX_HIDDEN) return TT_ERR_SIZE;
  if (!x_bf16 || !router_w_bf16 || !gate_up_packed || !down_packed || !out_bf16 || !out_idx ||
      !out_prob)
    return TT_ERR_NULL;
  if (!aligned(x_bf16, 16) || !aligned(router_w_bf16, 16) || !aligned(gate_up_packed, 8) ||
      !aligned(down_packed, 8) || !aligned(out_bf16, 2) || !aligned(out_idx, 4) ||
      !aligned(out_prob, 4))
    return TT_ERR_ALIGN;
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  cudaError_t e = tt::moe_static_scratch(&scratch, &scratch_bytes);
  if (e != cudaSuccess) return from_cuda(e);
  if (scratch_bytes < tt_moe_workspace_bytes(hidden, inter, n_experts, top_k)) return TT_ERR_SIZE;
  e = tt::launch_moe(x_bf16, int(hidden), int(inter), router_w_bf16, int(n_experts), int(top_k),
                     reinterpret_cast<const uint8_t* const*>(gate_up_packed),
                     reinterpret_cast<const uint8_t* const*>(down_packed), out_bf16, out_idx,
                     out_prob, scratch, as_stream(stream), kPdl);
  if (e == cudaErrorInvalidConfiguration) return TT_ERR_UNSUPPORTED;
  return from_cuda(e);
}

tt_status tt_quantize_fp8(const float* w, int64_t n, int64_t k, uint8_t* codes, float* scales,
                          int32_t* status_dev, void* stream) {
  if (n < 0 || k < 0 || n > kMaxRows) return TT_ERR_SHAPE;
  if (n == 0 || k == 0) return TT_OK;
  if (!w || !codes || !scales) return TT_ERR_NULL;
  if (!aligned(w, 4) || !aligned(scales, 4) || (status_dev && !aligned(status_dev, 4)))
    return TT_ERR_ALIGN;
  return from_cuda(tt::launch_quantize_fp8(w, n, k, codes, scales, status_dev, as_stream(stream)));
}

namespace {
inline tt_status fp8_shape(int64_t n, int64_t k, int64_t m) {
  if (n < 1 || n > kMaxRows || k < 16 || k % 16 != 0 || k > kMaxK) return TT_ERR_SHAPE;
  if (m < 1 || m > 8) return TT_ERR_SHAPE;
  return TT_OK;
}
}  // namespace

tt_status tt_fp8_matvec(const uint8_t* codes, const float* scales, int64_t n, int64_t k,
                        const uint16_t* x_bf16, int64_t m, uint16_t* y_bf16, void* stream) {
  if (tt_status st = fp8_shape(n, k, m)) return st;
  if (!codes || !scales || !x_bf16 || !y_bf16) return TT_ERR_NULL;
  if (!aligned(codes, 16) || !aligned(scales, 4) || !aligned(x_bf16, 16) || !aligned(y_bf16, 2))
    return TT_ERR_ALIGN;
  const cudaError_t e = tt::launch_fp8_matvec(codes, scales, int(n), int(k), x_bf16, int(m),
                                              y_bf16, as_stream(stream), kPdl);
  if (e == cudaErrorInvalidConfiguration) return TT_ERR_UNSUPPORTED;
  return from_cuda(e);
}

tt_status tt_fp8_swiglu_matvec(const uint8_t* gate_codes, const float* gate_scales,
                               const uint8_t* up_codes, const float* up_scales, int64_t n,
                               int64_t k, const uint16_t* x_bf16, int64_t m, uint16_t* h_bf16,
                               void* stream) {
  if (tt_status st = fp8_shape(n, k, m)) return st;
  if (!gate_codes || !gate_scales || !up_codes || !up_scales || !x_bf16 || !h_bf16)
    return TT_ERR_NULL;
  if (!aligned(gate_codes, 16) || !aligned(up_codes, 16) || !aligned(gate_scales, 4) ||
      !aligned(up_scales, 4) || !aligned(x_bf16, 16) || !aligned(h_bf16, 2))
    return TT_ERR_ALIGN;
  const cudaError_t e = tt::launch_fp8_swiglu(gate_codes, gate_scales, up_codes, up_scales,
                                              int(n), int(k), x_bf16, int(m), h_bf16,
                                              as_stream(stream), kPdl);
  if (e == cudaErrorInvalidConfiguration) return TT_ERR_UNSUPPORTED;
  return from_cuda(e);
}

tt_status tt_quantize_int4_grouped(const float* w, int64_t n, int64_t k, int32_t group,
                                   uint8_t* codes, uint16_t* scales_f16, uint8_t* zp_u4,
                                   int32_t* status_dev, void* stream) {
  if (n < 0 || k < 0 || k % 2 != 0 || group < 2 || group % 2 != 0 || n > kMaxRows)
    return TT_ERR_SHAPE;
  if (n == 0 || k == 0) return TT_OK;
  if (!w || !codes || !scales_f16 || !zp_u4) return TT_ERR_NULL;
  if (!aligned(w, 4) || !aligned(scales_f16, 2) || (status_dev && !aligned(status_dev, 4)))
    return TT_ERR_ALIGN;
  return from_cuda(tt::launch_quantize_int4(w, n, k, group, codes, scales_f16, zp_u4, status_dev,
                                            as_stream(stream)));
}

tt_status tt_int4_grouped_matvec(const uint8_t* codes, const uint16_t* scales_f16,
                                 const uint8_t* zp_u4, int64_t n, int64_t k, int32_t group,
                                 const uint16_t* x_bf16, int64_t m, uint16_t* y_bf16,
                                 void* stream) {
  if (n < 1 || k < 32 || k % 32 != 0 || k > 8192 || n > kMaxRows) return TT_ERR_SHAPE;
  if (group < 32 || group % 32 != 0) return TT_ERR_SHAPE;
  if (m < 1 || m > 8) return TT_ERR_SHAPE;
  if (!codes || !scales_f16 || !zp_u4 || !x_bf16 || !y_bf16) return TT_ERR_NULL;
  if (!aligned(codes, 16) || !aligned(scales_f16, 2) || !aligned(x_bf16, 16) ||
      !aligned(y_bf16, 2))
    return TT_ERR_ALIGN;
  const cudaError_t e = tt::launch_int4_matvec(codes, scales_f16, zp_u4, int(n), int(k),
                                               int(group), x_bf16, int(m), y_bf16,
                                               as_stream(stream), kPdl);
  if (e == cudaErrorInvalidConfiguration) return TT_ERR_UNSUPPORTED;
  return from_cuda(e);
}

size_t tt_gqa_decode_workspace_bytes(int32_t heads, int32_t kv_heads, int32_t head_dim) {
  if (heads < 1 || kv_heads < 1 || heads % kv_heads != 0) return 0;
  if (head_dim != 64 && head_dim != 128) return 0;
  if (heads / kv_heads > 16 || kv_heads > tt::kGqaMaxKvHeads) return 0;
  return tt::gqa_decode_workspace_bytes(heads, kv_heads, head_dim);
}

tt_status tt_gqa_decode_attention(const uint16_t* q_bf16, const uint16_t* k_cache,
                                  const uint16_t* v_cache, int32_t heads, int32_t kv_heads,
                                  int32_t head_dim, int64_t cap, int64_t len, float scale,
                                  uint16_t* out_bf16, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  if (heads < 1 || kv_heads < 1 || heads % kv_heads != 0 || head_dim < 1) return TT_ERR_SHAPE;
  if (len < 1 || cap < len) return TT_ERR_SHAPE;
  if (!std::isfinite(scale)) return TT_ERR_NONFINITE;
  if (cap > (int64_t(1) << 31)) return TT_ERR_UNSUPPORTED;  // TMA coordinates and strides
  if (head_dim != 64 && head_dim != 128) return TT_ERR_UNSUPPORTED;
  if (heads / kv_heads > 16 || kv_heads > tt::kGqaMaxKvHeads) return TT_ERR_UNSUPPORTED;
  if (!q_bf16 || !k_cache || !v_cache || !out_bf16 || !workspace) return TT_ERR_NULL;
  if (workspace_bytes < tt::gqa_decode_workspace_bytes(heads, kv_heads, head_dim))
    return TT_ERR_SIZE;
  if (!aligned(q_bf16, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(out_bf16, 16) || !aligned(workspace, 16))
    return TT_ERR_ALIGN;
  const cudaError_t e =
      tt::launch_gqa_decode(q_bf16, k_cache, v_cache, heads, kv_heads, head_dim, cap, len, scale,
                            out_bf16, workspace, as_stream(stream), kPdl);
  if (e == cudaErrorInvalidConfiguration) return TT_ERR_UNSUPPORTED;
  return from_cuda(e);
}

size_t tt_lowbit_matrix_bytes(int32_t bits, int64_t n, int64_t k) {
  if ((bits != 1 && bits != 2) || n < 1 || k < 1 || n > kMaxRows || k > (int64_t(1) << 30))
    return 0;
  return tt::lowbit_matrix_bytes(bits, n, k);
}

tt_status tt_quantize_lowbit(int32_t bits, const float* w, int64_t n, int64_t k, void* buf,
                             size_t buf_bytes, int32_t* status_dev, void* stream) {
  if (bits != 1 && bits != 2) return TT_ERR_SHAPE;
  if (n < 0 || k < 1 || n > kMaxRows || k > (int64_t(1) << 30)) return TT_ERR_SHAPE;
  if (n == 0) return TT_OK;
  if (!w || !buf) return TT_ERR_NULL;
  if (buf_bytes < tt::lowbit_matrix_bytes(bits, n, k)) return TT_ERR_SIZE;
  if (!aligned(w, 4) || !aligned(buf, 16) || (status_dev && !aligned(status_dev, 4)))
    return TT_ERR_ALIGN;
  return from_cuda(tt::launch_quantize_lowbit(bits, w, n, k, static_cast<uint8_t*>(buf),
                                              status_dev, as_stream(stream)));
}

size_t tt_moe_lowbit_workspace_bytes(int64_t inter, int32_t n_experts, int32_t top_k) {
  if (inter < 32 || inter > 8192 || n_experts < 1 || n_experts > 256 || top_k < 1 ||
      top_k > 8 || top_k > n_experts)
    return 0;
  return size_t(top_k) * size_t(inter) * 4 + (size_t(n_experts) * 4 + 15) / 16 * 16;
}

tt_status tt_moe_lowbit_topk_mlp(int32_t bits, const uint16_t* x_bf16, int64_t hidden,
                                 int64_t inter, const uint16_t* router_w_bf16, int32_t n_experts,
                                 int32_t top_k, const void* const* gate_up,
                                 const void* const* down, uint16_t* out_bf16, int32_t* out_idx,
                                 float* out_prob, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  if (bits != 1 && bits != 2) return TT_ERR_SHAPE;
  if (hidden < 32 || hidden % 32 != 0 || hidden > 8192) return TT_ERR_SHAPE;
  if (inter < 32 || inter % 32 != 0 || inter > 8192) return TT_ERR_SHAPE;
  if (n_experts < 1 || n_experts > 256 || top_k < 1 || top_k > 8 || top_k > n_experts)
    return TT_ERR_SHAPE;
  if (!x_bf16 || !router_w_bf16 || !gate_up || !down || !out_bf16 || !out_idx || !out_prob ||
      !workspace)
    return TT_ERR_NULL;
  if (workspace_bytes < tt_moe_lowbit_workspace_bytes(inter, n_experts, top_k)) return TT_ERR_SIZE;
  if (!aligned(x_bf16, 16) || !aligned(router_w_bf16, 16) || !aligned(gate_up, 8) ||
      !aligned(down, 8) || !aligned(out_bf16, 2) || !aligned(out_idx, 4) ||
      !aligned(out_prob, 4) || !aligned(workspace, 16))
    return TT_ERR_ALIGN;
  const cudaError_t e = tt::launch_moe_lowbit(
      bits, x_bf16, int(hidden), int(inter), router_w_bf16, n_experts, top_k,
      reinterpret_cast<const uint8_t* const*>(gate_up),
      reinterpret_cast<const uint8_t* const*>(down), out_bf16, out_idx, out_prob, workspace,
      as_stream(stream), kPdl);
  if (e == cudaErrorInvalidConfiguration) return TT_ERR_UNSUPPORTED;
  return from_cuda(e);
}

}  // extern "C"
