// Setup-time kernels: MXFP4 and grouped INT4 quantisers, the MXFP4 test-aid
// dequantiser and the loaders that rearrange canonical MXFP4 bytes into the
// packed record layouts of layout.cuh.
//
// Quantiser rules follow the production MXFP4 / INT4 quantizers of the
// ThinTensor project page (stardance.hackclub.com/projects/29750, "Hitting
// 100hrs and final ship"; "correct affine INT4 partial-group quantization"
// in the fixes list).  The GPU side takes each rounding decision with the
// hardware conversions (cvt.rn.satfinite.e2m1x2.f32, cvt.rn.f16.f64), which
// the parity tests compare bit for bit against an independent CPU oracle.
#include "common.cuh"
#include "launch.h"
#include "layout.cuh"

namespace tt {

namespace {

// Two fp32 values -> one byte of E2M1 codes (lo in bits 0..3, hi in 4..7),
// round to nearest even, saturating at +-6.  The sign bit is forced from the
// input so that negative values rounding to zero give code 0x8.
__device__ __forceinline__ uint32_t e2m1x2_from_f32(float lo, float hi) {
  uint32_t b;
  asm("{\n\t.reg .b8 r;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 r, %1, %2;\n\t"
      "cvt.u32.u8 %0, r;\n\t}"
      : "=r"(b)
      : "f"(hi), "f"(lo));
  b |= ((__float_as_uint(lo) >> 31) << 3) | ((__float_as_uint(hi) >> 31) << 7);
  return b & 0xFFu;
}

__global__ void quantize_mxfp4_kernel(const float* __restrict__ w, int64_t n, int64_t k,
                                      uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                      int32_t* status) {
  const int64_t nblk = k >> 5;
  const int64_t total = n * nblk;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / nblk, b = t - r * nblk;
    const float4* src = reinterpret_cast<const float4*>(w + r * k + b * 32);
    float v[32];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float4 f = src[q];
      v[4 * q + 0] = f.x;
      v[4 * q + 1] = f.y;
      v[4 * q + 2] = f.z;
      v[4 * q + 3] = f.w;
    }
    bool finite = true;
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      finite = finite && isfinite(v[i]);
      amax = fmaxf(amax, fabsf(v[i]));
    }
    uint32_t out[4] = {0u, 0u, 0u, 0u};
    uint32_t sbyte;
    if (!finite) {
      sbyte = 0xFFu;
      if (status) atomicOr(status, 4);  // TT_ERR_NONFINITE
    } else {
      // floor(log2 amax) from the exponent field; a zero or subnormal amax
      // lands on the clamp X = -127.
      const int ebits = int((__float_as_uint(amax) >> 23) & 0xFFu);
      const int X = (ebits == 0) ? -127 : max(ebits - 127 - 2, -127);
      sbyte = uint32_t(X + 127);
      const float inv = scalbnf(1.0f, -X);  // exact power of two
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        uint32_t byte = e2m1x2_from_f32(v[2 * j] * inv, v[2 * j + 1] * inv);
        out[j >> 2] |= byte << (8 * (j & 3));
      }
    }
    *reinterpret_cast<uint4*>(codes + r * (k >> 1) + b * 16) =
        make_uint4(out[0], out[1], out[2], out[3]);
    scales[r * nblk + b] = uint8_t(sbyte);
  }
}

__global__ void dequantize_mxfp4_kernel(const uint8_t* __restrict__ codes,
                                        const uint8_t* __restrict__ scales, int64_t n, int64_t k,
                                        float* __restrict__ out) {
  const int64_t half = k >> 1;
  const int64_t total = n * half;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / half, j = t - r * half;  // byte j of row r: k = 2j, 2j+1
    const uint32_t byte = codes[t];
    uint32_t h0, h1, h2, h3;
    e2m1x8_to_f16x2(byte, h0, h1, h2, h3);
    const uint32_t sb = scales[r * (k >> 5) + (2 * j) / 32];
    const float sc = (sb == 255u) ? __uint_as_float(0x7FC00000u) : e8m0_to_f32(sb);
    __half2 hv = *reinterpret_cast<__half2*>(&h0);
    float2 f = __half22float2(hv);
    *reinterpret_cast<float2*>(out + r * k + 2 * j) = make_float2(f.x * sc, f.y * sc);
  }
}

__global__ void pack_swiglu_kernel(const uint8_t* __restrict__ gc, const uint8_t* __restrict__ gs,
                                   const float* __restrict__ gp, const uint8_t* __restrict__ uc,
                                   const uint8_t* __restrict__ us, const float* __restrict__ up,
                                   int64_t n, int k, uint8_t* __restrict__ packed) {
  const SwigluRecord L(k);
  const int64_t total = n * L.bytes;
  const int half = k >> 1;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / L.bytes;
    const int o = int(t - r * L.bytes);
    uint32_t v = 0;
    if (o < half) {
      v = gc[r * half + o];
    } else if (o < k) {
      v = uc[r * half + (o - half)];
    } else if (o < k + L.nblk) {
      v = gs[r * L.nblk + (o - k)];
    } else if (o < k + 2 * L.nblk) {
      v = us[r * L.nblk + (o - k - L.nblk)];
    } else if (o >= L.post && o < L.post + 8) {
      const float* src = (o < L.post + 4) ? gp : up;
      const float f = src ? src[r] : 1.0f;
      v = (__float_as_uint(f) >> (8 * ((o - L.post) & 3))) & 0xFFu;
    }
    packed[t] = uint8_t(v);
  }
}

// One thread per output byte of the column-sliced layout (ColSlices).
__global__ void pack_rows_kernel(const uint8_t* __restrict__ codes,
                                 const uint8_t* __restrict__ scales, int64_t n, int k,
                                 uint8_t* __restrict__ packed) {
  const ColSlices L(n, k);
  const int half = k >> 1;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < L.bytes;
       t += (int64_t)gridDim.x * blockDim.x) {
    uint32_t v = 0;
    if (t < n * half) {  // codes: t = (slice * n + row) * 8 + byte
      const int64_t sr = t >> 3;
      const int sl = int(sr / n);
      const int64_t r = sr - (int64_t)sl * n;
      v = codes[r * half + sl * 8 + (t & 7)];
    } else if (t >= L.scales_off && t < L.scales_off + n * L.nblk) {
      const int64_t o = t - L.scales_off;  // block * n + row
      const int b = int(o / n);
      const int64_t r = o - (int64_t)b * n;
      v = scales[r * L.nblk + b];
    }
    packed[t] = uint8_t(v);
  }
}

// Grouped affine INT4.  One thread per (row, pair of groups) so that no two
// threads write the same zero-point byte.  The scale is computed in fp64 and
// rounded once to fp16 (cvt.rn.f16.f64); zp and q use rint (ties to even).
__device__ void int4_one_group(const float* __restrict__ wr, int64_t lo, int64_t hi,
                               uint8_t* __restrict__ cr, uint16_t* sdst, uint32_t* zp_nibble,
                               int32_t* status) {
  bool finite = true;
  float mn = wr[lo], mx = wr[lo];
  for (int64_t kk = lo; kk < hi; ++kk) {
    const float v = wr[kk];
    finite = finite && isfinite(v);
    mn = fminf(mn, v);
    mx = fmaxf(mx, v);
  }
  __half s16;
  if (!finite) {
    s16 = __ushort_as_half(0x7E00);
  } else {
    const double range = double(mx) - double(mn);
    s16 = __double2half(range / 15.0);
  }
  *sdst = __half_as_ushort(s16);
  const double s = double(__half2float(s16));
  *zp_nibble = 0;
  const bool bad = !finite || isinf(s);
  if (bad && status) atomicOr(status, 4);  // TT_ERR_NONFINITE
  double z = 0.0;
  const bool zero = bad || s == 0.0;
  if (!zero) z = fmin(fmax(rint(-double(mn) / s), 0.0), 15.0);
  *zp_nibble = uint32_t(z);
  for (int64_t kk = lo; kk < hi; kk += 2) {  // lo, hi even
    uint32_t q0 = 0, q1 = 0;
    if (!zero) {
      q0 = uint32_t(fmin(fmax(rint(double(wr[kk]) / s) + z, 0.0), 15.0));
      q1 = uint32_t(fmin(fmax(rint(double(wr[kk + 1]) / s) + z, 0.0), 15.0));
    }
    cr[kk >> 1] = uint8_t(q0 | (q1 << 4));
  }
}

__global__ void quantize_int4_kernel(const float* __restrict__ w, int64_t n, int64_t k, int group,
                                     uint8_t* __restrict__ codes, uint16_t* __restrict__ scales,
                                     uint8_t* __restrict__ zp, int32_t* status) {
  const int64_t ng = (k + group - 1) / group;
  const int64_t zb = (ng + 1) / 2;
  const int64_t total = n * zb;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / zb, p = t - r * zb;
    const float* wr = w + r * k;
    uint8_t* cr = codes + r * (k >> 1);
    uint32_t z0 = 0, z1 = 0;
    for (int h = 0; h < 2; ++h) {
      const int64_t g = 2 * p + h;
      if (g >= ng) break;
      const int64_t lo = g * group;
      const int64_t hi = min(lo + (int64_t)group, k);
      int4_one_group(wr, lo, hi, cr, scales + r * ng + g, h ? &z1 : &z0, status);
    }
    zp[r * zb + p] = uint8_t(z0 | (z1 << 4));
  }
}

int grid_for(int64_t work, int threads) {
  int64_t blocks = (work + threads - 1) / threads;
  if (blocks < 1) blocks = 1;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  return int(blocks);
}

}  // namespace

cudaError_t launch_quantize_mxfp4(const float* w, int64_t n, int64_t k, uint8_t* codes,
                                  uint8_t* scales, int32_t* status, cudaStream_t s) {
  const int64_t work = n * (k / 32);
  if (work == 0) return cudaSuccess;
  quantize_mxfp4_kernel<<<grid_for(work, 256), 256, 0, s>>>(w, n, k, codes, scales, status);
  return cudaGetLastError();
}

cudaError_t launch_dequantize_mxfp4(const uint8_t* codes, const uint8_t* scales, int64_t n,
                                    int64_t k, float* out, cudaStream_t s) {
  const int64_t work = n * (k / 2);
  if (work == 0) return cudaSuccess;
  dequantize_mxfp4_kernel<<<grid_for(work, 256), 256, 0, s>>>(codes, scales, n, k, out);
  return cudaGetLastError();
}

cudaError_t launch_pack_swiglu(const uint8_t* gc, const uint8_t* gs, const float* gp,
                               const uint8_t* uc, const uint8_t* us, const float* up, int64_t n,
                               int64_t k, uint8_t* packed, cudaStream_t s) {
  const int64_t work = n * SwigluRecord(int(k)).bytes;
  pack_swiglu_kernel<<<grid_for(work, 256), 256, 0, s>>>(gc, gs, gp, uc, us, up, n, int(k),
                                                         packed);
  return cudaGetLastError();
}

cudaError_t launch_pack_rows(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k,
                             uint8_t* packed, cudaStream_t s) {
  const int64_t work = ColSlices(n, int(k)).bytes;
  pack_rows_kernel<<<grid_for(work, 256), 256, 0, s>>>(codes, scales, n, int(k), packed);
  return cudaGetLastError();
}

cudaError_t launch_quantize_int4(const float* w, int64_t n, int64_t k, int group,
                                 uint8_t* codes, uint16_t* scales, uint8_t* zp, int32_t* status,
                                 cudaStream_t s) {
  const int64_t ng = (k + group - 1) / group;
  const int64_t work = n * ((ng + 1) / 2);
  if (work == 0) return cudaSuccess;
  quantize_int4_kernel<<<grid_for(work, 128), 128, 0, s>>>(w, n, k, group, codes, scales, zp,
                                                           status);
  return cudaGetLastError();
}

}  // namespace tt
