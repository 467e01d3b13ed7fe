// Internal launchers (host side).  Arguments are already validated by the
// C-ABI layer in api.cu; each returns the cudaError_t of its launch(es).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace tt {

struct DeviceInfo {
  int device = 0;
  int sms = 0;
  int smem_optin = 0;
  int32_t* error_word = nullptr;  // the library's device error word
};
// Cached per device; returns nullptr if the device cannot be queried.
const DeviceInfo* device_info();

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) only when a kernel needs
// more dynamic shared memory on this device than was already granted: the
// attribute call costs about a microsecond of host time, too much on the
// per-call path of kernels that take a few microseconds.
cudaError_t ensure_dynamic_smem(const void* kern, int device, int bytes);
template <typename Kern>
cudaError_t ensure_smem(const DeviceInfo& di, Kern kern, int bytes) {
  return ensure_dynamic_smem(reinterpret_cast<const void*>(kern), di.device, bytes);
}

// quantize.cu
cudaError_t launch_quantize_mxfp4(const float* w, int64_t n, int64_t k, uint8_t* codes,
                                  uint8_t* scales, int32_t* status, cudaStream_t s);
cudaError_t launch_dequantize_mxfp4(const uint8_t* codes, const uint8_t* scales, int64_t n,
                                    int64_t k, float* out, cudaStream_t s);
cudaError_t launch_pack_swiglu(const uint8_t* gc, const uint8_t* gs, const float* gp,
                               const uint8_t* uc, const uint8_t* us, const float* up,
                               int64_t n, int64_t k, uint8_t* packed, cudaStream_t s);
cudaError_t launch_pack_rows(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k,
                             uint8_t* packed, cudaStream_t s);
cudaError_t launch_quantize_int4(const float* w, int64_t n, int64_t k, int group,
                                 uint8_t* codes, uint16_t* scales, uint8_t* zp, int32_t* status,
                                 cudaStream_t s);

// gemv_mxfp4.cu — CUDA-core gate/up SwiGLU matvec, m in [1, 8]
cudaError_t launch_swiglu_mxfp4_cc(const uint8_t* packed, int n, int k, const uint16_t* x,
                                   int m, uint16_t* h, cudaStream_t s, bool pdl);

// gemv_mxfp4_mma.cu — gate/up SwiGLU with the multiply-adds on mma.sync, m in
// [2, 8], k <= 5120; otherwise cudaErrorInvalidConfiguration (nothing launched)
cudaError_t launch_swiglu_mxfp4_mma(const uint8_t* packed, int n, int k, const uint16_t* x,
                                    int m, uint16_t* h, cudaStream_t s, bool pdl);

// tc_swiglu.cu — tcgen05 gate/up SwiGLU, m in [1, 64] (the library sends
// m >= 4), k % 64 == 0; a plan that does not fit: cudaErrorInvalidConfiguration
cudaError_t launch_swiglu_mxfp4_tc(const uint8_t* packed, int n, int k, const uint16_t* x,
                                   int m, uint16_t* h, cudaStream_t s, bool pdl);
int tc_swiglu_smem_bytes(int m, int k);

// gemv_int4.cu — grouped affine INT4 matvec, m in [1, 8]
cudaError_t launch_int4_matvec(const uint8_t* codes, const uint16_t* scales, const uint8_t* zp,
                               int n, int k, int group, const uint16_t* x, int m, uint16_t* y,
                               cudaStream_t s, bool pdl);

// moe.cu / moe_fused.cu — router, top-k, the selected experts' gate/up and
// down as one cooperative kernel (moe_fused.cu); plan that does not fit the
// shared memory: cudaErrorInvalidConfiguration
size_t moe_workspace_bytes(int64_t hidden, int64_t inter, int n_experts, int top_k);
size_t moe_fused_workspace_bytes(int64_t hidden);
// gu, dn: device arrays of E device pointers (one packed buffer per expert)
cudaError_t launch_moe(const uint16_t* x, int hidden, int inter, const uint16_t* wr, int E,
                       int top_k, const uint8_t* const* gu, const uint8_t* const* dn,
                       uint16_t* out, int32_t* out_idx, float* out_prob, void* ws,
                       cudaStream_t s, bool pdl);
cudaError_t launch_moe_fused(const uint16_t* x, int hidden, int inter, const uint16_t* wr, int E,
                             int top_k, const uint8_t* const* gu, const uint8_t* const* dn,
                             uint16_t* out, int32_t* out_idx, float* out_prob, void* ws,
                             cudaStream_t s, bool pdl);
// The library-owned MoE scratch (a static device array) of the current
// device: its address (looked up on the first call on each device) and size.
constexpr int kMoeStaticMaxHidden = 4096;  // hidden limit of the static scratch
cudaError_t moe_static_scratch(void** ptr, size_t* bytes);

// fp8.cu — E4M3 weights with one fp32 scale per row: quantiser, matvec and
// gate/up SwiGLU (m in [1, 8]); x staging that does not fit the shared
// memory: cudaErrorInvalidConfiguration
cudaError_t launch_quantize_fp8(const float* w, int64_t n, int64_t k, uint8_t* codes,
                                float* scales, int32_t* status, cudaStream_t s);
cudaError_t launch_fp8_matvec(const uint8_t* codes, const float* scales, int n, int k,
                              const uint16_t* x, int m, uint16_t* y, cudaStream_t s, bool pdl);
cudaError_t launch_fp8_swiglu(const uint8_t* gc, const float* gs, const uint8_t* uc,
                              const float* us, int n, int k, const uint16_t* x, int m,
                              uint16_t* h, cudaStream_t s, bool pdl);

// gemv_rows.cu — single-matrix matvecs (dense down projection), m in [1, 8]:
// MXFP4 on canonical buffers (x staging that does not fit the shared memory:
// cudaErrorInvalidConfiguration) and bf16
cudaError_t launch_mxfp4_rows(const uint8_t* codes, const uint8_t* scales, const float* post,
                              int n, int k, const uint16_t* x, int m, uint16_t* y, cudaStream_t s,
                              bool pdl);
cudaError_t launch_bf16_rows(const uint16_t* w, int n, int k, const uint16_t* x, int m,
                             uint16_t* y, cudaStream_t s, bool pdl);

// attention.cu — single-token GQA over a bf16 KV cache, head_dim 64 or 128,
// up to 16 query heads per kv head, up to 64 kv heads; a split kernel writes
// per-split partials to the workspace, a merge kernel combines them.
constexpr int kGqaMaxKvHeads = 64;
constexpr int kGqaMaxSplits = 256;
size_t gqa_decode_workspace_bytes(int heads, int kv_heads, int head_dim);
cudaError_t launch_gqa_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v, int heads,
                              int kv_heads, int head_dim, int64_t cap, int64_t len, float scale,
                              uint16_t* out, void* ws, cudaStream_t s, bool pdl);

// moe_lowbit.cu — Q1 / Q2 low-bit experts: quantiser and the MoE layer
// (router, selected-expert SwiGLU, weighted down projection; three kernels).
// The workspace holds h fp32 [top_k][inter], then the E router logits.
size_t lowbit_matrix_bytes(int bits, int64_t n, int64_t k);
int lowbit_table_smem_bytes(int64_t k);
cudaError_t launch_quantize_lowbit(int bits, const float* w, int64_t n, int64_t k, uint8_t* buf,
                                   int32_t* status, cudaStream_t s);
cudaError_t launch_moe_lowbit(int bits, const uint16_t* x, int hidden, int inter,
                              const uint16_t* wr, int E, int top_k, const uint8_t* const* gu,
                              const uint8_t* const* dn, uint16_t* out, int32_t* out_idx,
                              float* out_prob, void* ws, cudaStream_t s, bool pdl);

// gemv_bf16.cu
cudaError_t launch_swiglu_bf16(const uint16_t* wg, const uint16_t* wu, int n, int k,
                               const uint16_t* x, int m, uint16_t* h, cudaStream_t s, bool pdl);

}  // namespace tt
