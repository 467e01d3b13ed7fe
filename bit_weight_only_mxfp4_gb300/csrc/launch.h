// Internal launchers (host side).  Arguments are already validated by the
// C-ABI layer in api.cu; each returns the cudaError_t of its launch(es).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace tt {

struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;
  int32_t* error_word = nullptr;  // the library's device error word
};
// Cached per device; returns nullptr if the device cannot be queried.
const DeviceInfo* device_info();

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

// gemv_mxfp4.cu — CUDA-core gate/up SwiGLU matvec, m in [1, 16]
cudaError_t launch_swiglu_mxfp4_cc(const uint8_t* packed, int n, int k, const uint16_t* x,
                                   int m, uint16_t* h, cudaStream_t s, bool pdl);

// gemv_bf16.cu
cudaError_t launch_swiglu_bf16(const uint16_t* wg, const uint16_t* wu, int n, int k,
                               const uint16_t* x, int m, uint16_t* h, cudaStream_t s, bool pdl);

}  // namespace tt
