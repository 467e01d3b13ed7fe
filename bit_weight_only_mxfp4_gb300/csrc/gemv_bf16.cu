// bf16 gate/up SwiGLU matvec for the layers a selective profile keeps in
// bf16 (ThinTensor devlog, kerbin.cskartikey.dev/@satvikhardat, Dev Log #4,
// "Why this was not just normal quantization": MXFP4 only on gate/up of
// layers 0:24, everything else bf16).
//
// At 2 bytes per weight the kernel is far from any ALU limit, so it streams
// the rows with plain 128-bit loads (eight per lane in flight per row),
// reads x through L1 with coherent loads (never the read-only path: x is
// the previous kernel's output, written while this kernel may already be
// resident), multiplies with fma.rn.f32.bf16 (bf16 x bf16 is exact
// in fp32) and reduces each row pair with one warp-shuffle pass.
#include "common.cuh"
#include "launch.h"

namespace tt {
namespace {

constexpr int kWarps = 8;
constexpr int kU = 8;  // 16-byte chunks per lane per row per step
constexpr int kBf16StageBytes = 48 * 1024;  // x staged in shared memory up to this size

__device__ __forceinline__ void fma8(float& a0, float& a1, const uint4& w, const uint4& xv) {
  fma_bf16x2_f32(a0, a1, w.x, xv.x);
  fma_bf16x2_f32(a0, a1, w.y, xv.y);
  fma_bf16x2_f32(a0, a1, w.z, xv.z);
  fma_bf16x2_f32(a0, a1, w.w, xv.w);
}

// How x is read (x is the previous kernel's output, so only with coherent
// loads, after the dependency wait):
//   kXRegs  m = 1 and k <= 32 * 8 * kU: each lane holds its chunks of x in
//           registers (one 128-bit load each) for every row;
//   kXSmem  x (m rows) copied once per CTA into shared memory, every row
//           reads it there;
//   kXL1    every row reads it through L1.
enum XMode { kXL1 = 0, kXSmem = 1, kXRegs = 2 };

template <int MT, int XM>
__global__ void __launch_bounds__(kWarps * 32, 2)
    swiglu_bf16_kernel(const uint16_t* __restrict__ wg, const uint16_t* __restrict__ wu, int n,
                       int k, const uint16_t* __restrict__ x, int m, uint16_t* __restrict__ h) {
  static_assert(XM != kXRegs || MT == 1, "x in registers for one batch row");
  constexpr bool STAGED = XM == kXSmem;
  extern __shared__ __align__(16) uint4 xsm[];  // kXSmem: x[i] at chunks i * cpr ..
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int nw = gridDim.x * kWarps;
  const int cpr = k >> 3;  // 16-byte chunks per row
  const uint4* x4 = reinterpret_cast<const uint4*>(x);
  auto load = [&](int r, int c0, uint4 (&gv)[kU], uint4 (&uv)[kU]) {
    const uint4* g4 = reinterpret_cast<const uint4*>(wg + (size_t)r * k);
    const uint4* u4 = reinterpret_cast<const uint4*>(wu + (size_t)r * k);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int c = c0 + u * 32 + lane;
      if (c < cpr) {
        gv[u] = __ldcs(g4 + c);
        uv[u] = __ldcs(u4 + c);
      } else {
        gv[u] = uv[u] = make_uint4(0, 0, 0, 0);
      }
    }
  };
  uint4 gv[kU], uv[kU];
  pdl_allow_next_grid();
  if (gw < n) load(gw, 0, gv, uv);  // weights do not depend on the producer of x
  pdl_wait_prior_grid();
  if (STAGED) {
    for (int t = threadIdx.x; t < m * cpr; t += kWarps * 32) xsm[t] = __ldcg(x4 + t);
    __syncthreads();
  }
  uint4 xr[kU];  // kXRegs: this lane's chunks 32 u + lane of x
  if (XM == kXRegs) {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int c = u * 32 + lane;
      xr[u] = c < cpr ? __ldcg(x4 + c) : make_uint4(0, 0, 0, 0);
    }
  }
  for (int r = gw; r < n; r += nw) {
    float ag0[MT], ag1[MT], au0[MT], au1[MT];
#pragma unroll
    for (int i = 0; i < MT; ++i) ag0[i] = ag1[i] = au0[i] = au1[i] = 0.f;
    for (int c0 = 0; c0 < cpr; c0 += 32 * kU) {
      if (r != gw || c0 != 0) load(r, c0, gv, uv);  // the first step is already in flight
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < cpr) {
#pragma unroll
          for (int i = 0; i < MT; ++i) {
            if (i < m) {
              const uint4 xv = XM == kXRegs ? xr[u]
                               : STAGED      ? xsm[(size_t)i * cpr + c]
                                             : __ldca(x4 + (size_t)i * cpr + c);
              fma8(ag0[i], ag1[i], gv[u], xv);
              fma8(au0[i], au1[i], uv[u], xv);
            }
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      const float v = warp_sum2(ag0[i] + ag1[i], au0[i] + au1[i], lane);
      const float vu = __shfl_sync(0xffffffffu, v, 16);
      if (lane == 0 && i < m) {
        __nv_bfloat16 b = __float2bfloat16_rn(silu_mul(v, vu));
        h[(size_t)i * n + r] = *reinterpret_cast<uint16_t*>(&b);
      }
    }
  }
}

template <int MT>
cudaError_t run(const DeviceInfo& di, const uint16_t* wg, const uint16_t* wu, int n, int k,
                const uint16_t* x, int m, uint16_t* h, cudaStream_t s, bool pdl) {
  int grid = 2 * di.sms;
  const int need = (n + kWarps - 1) / kWarps;
  if (grid > need) grid = need;
  cudaLaunchConfig_t cfg = {};
  // x in registers for one batch row of at most 32 * 8 * kU values, else in
  // shared memory when it fits beside a second CTA on the SM
  const int xbytes = m * k * 2;
  const bool regs = MT == 1 && k <= 32 * 8 * kU;
  const bool staged = !regs && xbytes <= kBf16StageBytes;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = staged ? xbytes : 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if constexpr (MT == 1)
    if (regs) return cudaLaunchKernelEx(&cfg, swiglu_bf16_kernel<1, kXRegs>, wg, wu, n, k, x, m, h);
  if (staged) return cudaLaunchKernelEx(&cfg, swiglu_bf16_kernel<MT, kXSmem>, wg, wu, n, k, x, m, h);
  return cudaLaunchKernelEx(&cfg, swiglu_bf16_kernel<MT, kXL1>, wg, wu, n, k, x, m, h);
}

}  // namespace

cudaError_t launch_swiglu_bf16(const uint16_t* wg, const uint16_t* wu, int n, int k,
                               const uint16_t* x, int m, uint16_t* h, cudaStream_t s, bool pdl) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorNoDevice;
  if (m == 1) return run<1>(*di, wg, wu, n, k, x, m, h, s, pdl);
  if (m == 2) return run<2>(*di, wg, wu, n, k, x, m, h, s, pdl);
  if (m <= 4) return run<4>(*di, wg, wu, n, k, x, m, h, s, pdl);
  return run<8>(*di, wg, wu, n, k, x, m, h, s, pdl);
}

}  // namespace tt
