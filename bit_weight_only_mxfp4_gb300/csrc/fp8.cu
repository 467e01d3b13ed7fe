// FP8 (E4M3) weights with one fp32 scale per row: quantiser, matvec and the
// gate/up SwiGLU matvec.
//
// Method: ThinTensor devlog (kerbin.cskartikey.dev/@satvikhardat), Dev Log #3
// "SmolLM3-3B Results": the quality FP8 profile keeps gate/up and the middle
// down projections in FP8, and its scaled matvec sums code value times x
// along the row and multiplies the sum by the row's scale.  The element
// format and the scale rule are not printed there; this library takes E4M3
// without infinities (largest magnitude 448) and scale = fp32(amax / 448).
//
// Matvec design.  With one scale per row there is no per-block factor, so
// the whole row can accumulate inside the tensor core (mma.sync m16n8k16,
// f16 x f16 -> fp32):
//  * a warp streams a pair of weight rows (gate and up, or rows r and r+1),
//    or a slice of the pair's K when rows are few and long, with plain
//    128-bit loads, double-buffered steps;
//  * a 512-byte group of a row splits into 8 chunks of 64 k (chunk g = the
//    bytes of lanes 4g..4g+3); in each of 4 MMAs, A row g holds 16 k of
//    chunk g of the first row and A row 8 + g the same k of the second row,
//    and B column c holds x of chunk c at chunk c's k and zeros elsewhere.
//    D[c][c] and D[8 + c][c] then accumulate the two rows' dot products over
//    chunk c; the other entries of D are never read.  Thread (g, t) reads the
//    16 bytes 64g + 16t .. +15 of each row with one load, decoded by
//    cvt.rn.f16x2.e4m3x2 (two codes per instruction);
//  * x is staged once per CTA in shared memory, in that fragment order, as
//    f16 after one exact power-of-two prescale per batch row (the row's max
//    |x| -> [2^14, 2^15), so every finite value fits);
//  * the diagonal entries meet in one warp reduction; the epilogue applies
//    2^-s, the row scale and (gate/up) silu(g) * u, and stores bf16.
// e4m3 x f16 products are exact; the tensor core accumulates in fp32.
#include <cmath>

#include "common.cuh"
#include "launch.h"
#include "mxfp4_core.cuh"

namespace tt {
namespace {

constexpr int kQThreads = 256;

// E4M3 code of t, round to nearest with ties to the even mantissa,
// saturating at 448, sign kept on zero; computed from the fp64 value (no
// intermediate rounding).
__device__ uint32_t e4m3_from_double(double t) {
  if (isnan(t)) return 0x7Fu;
  const uint32_t sign = signbit(t) ? 0x80u : 0u;
  const double a = fabs(t);
  if (a >= 448.0) return sign | 0x7Eu;
  if (a < 0.015625) {                       // below 2^-6: steps of 2^-9
    return sign | uint32_t(rint(a * 512.0));  // 8 = 2^-6 = code 0x08
  }
  int e2;
  (void)frexp(a, &e2);  // a = f * 2^e2, f in [0.5, 1)
  int E = e2 - 1;       // a in [2^E, 2^(E+1))
  double q = rint(ldexp(a, 3 - E));  // in [8, 16]
  if (q == 16.0) {
    q = 8.0;
    ++E;
  }
  return sign | (uint32_t(E + 7) << 3) | (uint32_t(q) - 8u);
}

// One warp per row: amax, the row's fp32 scale, then every code.
__global__ void __launch_bounds__(kQThreads)
    quantize_fp8_kernel(const float* __restrict__ w, int64_t n, int64_t k,
                        uint8_t* __restrict__ codes, float* __restrict__ scales,
                        int32_t* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * (kQThreads / 32) + (threadIdx.x >> 5);
  if (r >= n) return;
  const float* wr = w + r * k;
  uint8_t* cr = codes + r * k;
  float amax = 0.f;
  bool finite = true;
  for (int64_t i = lane; i < k; i += 32) {
    const float v = wr[i];
    finite = finite && isfinite(v);
    amax = fmaxf(amax, fabsf(v));
  }
  amax = warp_max(amax);
  finite = __all_sync(0xffffffffu, finite);
  if (!finite) {
    for (int64_t i = lane; i < k; i += 32) cr[i] = 0;
    if (lane == 0) {
      scales[r] = __int_as_float(0x7FC00000);
      if (status) atomicOr(status, kErrNonfinite);
    }
    return;
  }
  const float s = __double2float_rn((double)amax / 448.0);
  if (lane == 0) scales[r] = s;
  if (s == 0.f) {  // amax = 0, or below what an fp32 scale can hold
    for (int64_t i = lane; i < k; i += 32) cr[i] = 0;
    return;
  }
  const double sd = (double)s;
  for (int64_t i = lane; i < k; i += 32) cr[i] = uint8_t(e4m3_from_double((double)wr[i] / sd));
}

// Two E4M3 codes per 16-bit half -> f16x2 (the lower byte in the low half).
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

constexpr int kWarps = 8;
constexpr int kGroupsPerStep = 4;  // 512-byte groups per row in flight per step

// MT: batch rows staged (m <= MT); SWIGLU: the row pair is (gate, up) of
// one output, else rows (2p, 2p + 1) of one matrix.
// ks warps share a pair (a down projection has few, long rows): the CTA's
// 8 warps take 8 / ks pairs at a time, warp (lp, sl) the sl-th slice of the
// groups of pair pb + lp; the slices' sums meet in shared memory and are
// added in slice order.
template <int MT, bool SWIGLU>
__global__ void __launch_bounds__(kWarps * 32, 2)
    fp8_pair_kernel(const uint8_t* __restrict__ wa, const float* __restrict__ sa,
                    const uint8_t* __restrict__ wb, const float* __restrict__ sb, int n, int k,
                    const uint16_t* __restrict__ x, int m, uint16_t* __restrict__ y, int ks) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float red[kWarps][MT][2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ngrp = (k + 511) >> 9;
  const int R = kWarps / ks, lp = warp / ks, sl = warp % ks;
  const int gs = (ngrp + ks - 1) / ks;  // groups per slice
  const int gbeg = sl * gs, gend = min(ngrp, gbeg + gs);
  uint4* xf = reinterpret_cast<uint4*>(smem);  // [MT][ngrp][32 lanes][2] f16 fragments
  int* sx = reinterpret_cast<int*>(xf + (size_t)MT * ngrp * 64);  // [MT] prescale exponents
  unsigned* xmax = reinterpret_cast<unsigned*>(sx + MT);            // [MT] max |x| bits
  const int npairs = SWIGLU ? n : (n + 1) / 2;
  const int pstep = gridDim.x * R;
  const int g = lane >> 2, t = lane & 3;

  pdl_allow_next_grid();
  // The first pair's first step of weights does not depend on the previous
  // kernel: request it before waiting.
  auto load_step = [&](int p, int q0, uint4 (&ca)[kGroupsPerStep], uint4 (&cb)[kGroupsPerStep]) {
    const int ra = SWIGLU ? p : 2 * p, rb = SWIGLU ? p : 2 * p + 1;
    const uint8_t* pa = wa + (size_t)ra * k;
    const uint8_t* pb = (SWIGLU || rb < n) ? wb + (size_t)rb * k : nullptr;
#pragma unroll
    for (int u = 0; u < kGroupsPerStep; ++u) {
      const int off = (q0 + u) * 512 + 16 * lane;
      ca[u] = cb[u] = make_uint4(0u, 0u, 0u, 0u);
      if (p < npairs && q0 + u < gend && off < k) {
        ca[u] = __ldcs(reinterpret_cast<const uint4*>(pa + off));
        if (pb) cb[u] = __ldcs(reinterpret_cast<const uint4*>(pb + off));
      }
    }
  };
  uint4 ca[kGroupsPerStep], cb[kGroupsPerStep];
  load_step(blockIdx.x * R + lp, gbeg, ca, cb);
  pdl_wait_prior_grid();

  // x: per batch row, the max |x| (bits of a non-negative float order like
  // the values), then the prescaled f16 fragments.
  if (threadIdx.x < MT) xmax[threadIdx.x] = 0u;
  __syncthreads();
  for (int i = 0; i < m; ++i) {
    float mx = 0.f;
    for (int c0 = 0; c0 < k / 8; c0 += 4 * kWarps * 32) {  // four loads in flight
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * kWarps * 32 + threadIdx.x;
        v[u] = c < k / 8 ? __ldca(reinterpret_cast<const uint4*>(x + (size_t)i * k + 8 * c))
                         : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t vw[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          mx = fmaxf(mx, fmaxf(fabsf(bf16_bits_to_f32(vw[e] & 0xFFFFu)),
                               fabsf(bf16_bits_to_f32(vw[e] >> 16))));
      }
    }
    mx = warp_max(mx);
    if (lane == 0) atomicMax(&xmax[i], __float_as_uint(mx));
  }
  __syncthreads();
  if (threadIdx.x < MT) {
    const float mx = __uint_as_float(xmax[threadIdx.x]);
    sx[threadIdx.x] = threadIdx.x < m && mx > 0.f ? min(f16_prescale_exponent(mx), 127) : 0;
  }
  __syncthreads();
  // fragment (i, q, l): x[i][512 q + 16 l .. +15] as 8 f16x2 (2 uint4)
  for (int it = threadIdx.x; it < MT * ngrp * 32; it += kWarps * 32) {
    const int i = it / (ngrp * 32), rem = it - i * ngrp * 32;
    const int off = (rem >> 5) * 512 + 16 * (rem & 31);
    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
    if (i < m && off < k) {
      v0 = __ldca(reinterpret_cast<const uint4*>(x + (size_t)i * k + off));
      v1 = __ldca(reinterpret_cast<const uint4*>(x + (size_t)i * k + off + 8));
    }
    const float two_s = scalbnf(1.0f, sx[i]);
    uint4 o0, o1;
    o0.x = pack_f16x2_scaled(bf16_bits_to_f32(v0.x & 0xFFFFu), bf16_bits_to_f32(v0.x >> 16), two_s);
    o0.y = pack_f16x2_scaled(bf16_bits_to_f32(v0.y & 0xFFFFu), bf16_bits_to_f32(v0.y >> 16), two_s);
    o0.z = pack_f16x2_scaled(bf16_bits_to_f32(v0.z & 0xFFFFu), bf16_bits_to_f32(v0.z >> 16), two_s);
    o0.w = pack_f16x2_scaled(bf16_bits_to_f32(v0.w & 0xFFFFu), bf16_bits_to_f32(v0.w >> 16), two_s);
    o1.x = pack_f16x2_scaled(bf16_bits_to_f32(v1.x & 0xFFFFu), bf16_bits_to_f32(v1.x >> 16), two_s);
    o1.y = pack_f16x2_scaled(bf16_bits_to_f32(v1.y & 0xFFFFu), bf16_bits_to_f32(v1.y >> 16), two_s);
    o1.z = pack_f16x2_scaled(bf16_bits_to_f32(v1.z & 0xFFFFu), bf16_bits_to_f32(v1.z >> 16), two_s);
    o1.w = pack_f16x2_scaled(bf16_bits_to_f32(v1.w & 0xFFFFu), bf16_bits_to_f32(v1.w >> 16), two_s);
    xf[2 * it] = o0;
    xf[2 * it + 1] = o1;
  }
  __syncthreads();

  const bool diag = (t == (g >> 1));  // holds D[g][g] and D[8 + g][g]
  const bool odd = (g & 1) != 0;
  uint4 wa2[kGroupsPerStep], wb2[kGroupsPerStep];  // the second step buffer
  for (int pb = blockIdx.x * R; pb < npairs; pb += pstep) {  // uniform over the CTA
    const int p = pb + lp;
    float d[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) d[i][0] = d[i][1] = d[i][2] = d[i][3] = 0.f;
    auto compute = [&](const uint4 (&xa)[kGroupsPerStep], const uint4 (&xb)[kGroupsPerStep],
                       int q0) {
#pragma unroll
      for (int u = 0; u < kGroupsPerStep; ++u) {
        const int q = q0 + u;
        if (q < gend) {
          const uint32_t wa4[4] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w};
          const uint32_t wb4[4] = {xb[u].x, xb[u].y, xb[u].z, xb[u].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // MMA j: bytes 4j..4j+3 of the thread's 16
            uint32_t a0, a2, b0, b2;
            e4m3x4_to_f16x2(wa4[j], a0, a2);
            e4m3x4_to_f16x2(wb4[j], b0, b2);
#pragma unroll
            for (int i = 0; i < MT; ++i) {
              if (i < m) {
                const uint4 xv = xf[((size_t)(i * ngrp + q) * 32 + lane) * 2 + (j >> 1)];
                const uint32_t x0 = (j & 1) ? xv.z : xv.x, x1 = (j & 1) ? xv.w : xv.y;
                mma_16816(d[i], a0, b0, a2, b2, x0, x1);
              }
            }
          }
        }
      }
    };
    // steps double-buffered: one step's loads in flight while the previous
    // one is computed; the next pair's first step follows the last
    for (int q0 = gbeg;; q0 += 2 * kGroupsPerStep) {
      const bool has_w = q0 + kGroupsPerStep < gend;
      if (has_w) load_step(p, q0 + kGroupsPerStep, wa2, wb2);
      if (p < npairs) compute(ca, cb, q0);
      const bool more = q0 + 2 * kGroupsPerStep < gend;
      if (more) load_step(p, q0 + 2 * kGroupsPerStep, ca, cb);
      else load_step(p + pstep, gbeg, ca, cb);
      if (has_w && p < npairs) compute(wa2, wb2, q0 + kGroupsPerStep);
      if (!more) break;
    }
    auto store = [&](int pp, int i, float v, float vu) {
      const int ra = SWIGLU ? pp : 2 * pp;
      const float fa = sa[ra];
      const float fb = SWIGLU ? sb[pp] : (2 * pp + 1 < n ? sb[2 * pp + 1] : 0.f);
      const float inv = scalbnf(1.0f, -sx[i]);
      const float ga = v * inv * fa, gb = vu * inv * fb;
      if (SWIGLU) {
        y[(size_t)i * n + pp] = f32_to_bf16_rne(silu_mul(ga, gb));
      } else {
        y[(size_t)i * n + 2 * pp] = f32_to_bf16_rne(ga);
        if (2 * pp + 1 < n) y[(size_t)i * n + 2 * pp + 1] = f32_to_bf16_rne(gb);
      }
    };
    if (ks == 1) {  // whole pairs per warp: no exchange
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const float va = diag ? (odd ? d[i][1] : d[i][0]) : 0.f;
        const float vb = diag ? (odd ? d[i][3] : d[i][2]) : 0.f;
        const float v = warp_sum2(va, vb, lane);  // lanes 0-15: first row, 16-31: second
        const float vu = __shfl_sync(0xffffffffu, v, 16);
        if (lane == 0 && p < npairs && i < m) store(p, i, v, vu);
      }
      continue;
    }
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      const float va = diag ? (odd ? d[i][1] : d[i][0]) : 0.f;
      const float vb = diag ? (odd ? d[i][3] : d[i][2]) : 0.f;
      const float v = warp_sum2(va, vb, lane);  // lanes 0-15: first row, 16-31: second
      if ((lane & 15) == 0) red[warp][i][lane >> 4] = v;
    }
    __syncthreads();
    if (threadIdx.x < R * MT) {
      const int lq = threadIdx.x / MT, i = threadIdx.x - lq * MT;
      const int pp = pb + lq;
      if (pp < npairs && i < m) {
        float v = 0.f, vu = 0.f;
        for (int s2 = 0; s2 < ks; ++s2) {
          v += red[lq * ks + s2][i][0];
          vu += red[lq * ks + s2][i][1];
        }
        store(pp, i, v, vu);
      }
    }
    __syncthreads();
  }
}

template <int MT, bool SWIGLU>
cudaError_t run_pair(const DeviceInfo& di, const uint8_t* wa, const float* sa, const uint8_t* wb,
                     const float* sb, int n, int k, const uint16_t* x, int m, uint16_t* y,
                     cudaStream_t s, bool pdl) {
  const int ngrp = (k + 511) / 512;
  const int smem = MT * ngrp * 64 * 16 + MT * 8;
  if (smem > di.smem_optin) return cudaErrorInvalidConfiguration;
  auto kern = fp8_pair_kernel<MT, SWIGLU>;
  cudaError_t e = ensure_smem(di, kern, smem);
  if (e != cudaSuccess) return e;
  const int npairs = SWIGLU ? n : (n + 1) / 2;
  // warps per pair: enough work items for a full grid several times over,
  // while a slice keeps at least 4 KB of the pair
  int ks = 1;
  while (ks < kWarps && (int64_t)npairs * ks < (int64_t)2 * 2 * di.sms * kWarps &&
         (int64_t)2 * k / (2 * ks) >= 4096)
    ks *= 2;
  int grid = 2 * di.sms;
  const int need = (npairs + kWarps / ks - 1) / (kWarps / ks);
  if (grid > need) grid = need;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, wa, sa, wb, sb, n, k, x, m, y, ks);
}

// Gate/up SwiGLU at m = 1 with K fixed at compile time (the gate/up layers
// of the models the library serves): a warp per row pair (gate row r, up
// row r), both rows' codes requested at once (KC / 512 chunks of 16 codes
// per lane and row), the warp's next pair in flight while the current one
// is computed, the first pair before the dependency wait.  x is staged once
// per CTA in shared memory with coherent loads after the wait: chunk c of
// the row (x[16 c .. 16 c + 15]) as f16 after an exact power-of-two prescale
// per chunk (its max |x| -> [2^14, 2^15)), kept as two arrays of 16-byte
// halves so a warp's reads are conflict-free, the inverse applied to the
// chunk's partial sums.  Codes are widened with cvt.rn.f16x2.e4m3x2 and
// multiplied by fma.rn.f32.f16 (exact products, fp32 sums); the row scales
// and SwiGLU follow the warp's reduction.
template <int KC>
__global__ void __launch_bounds__(kWarps * 32, 2)
    fp8_swiglu_k_kernel(const uint8_t* __restrict__ gc, const float* __restrict__ gs,
                        const uint8_t* __restrict__ uc, const float* __restrict__ us, int n,
                        const uint16_t* __restrict__ x, uint16_t* __restrict__ h) {
  static_assert(KC % 512 == 0, "whole 16-code chunks for every lane");
  constexpr int kU = KC / 512;    // chunks per lane and row
  constexpr int kCh = KC / 16;    // chunks per row
  __shared__ uint4 xlo[kCh], xhi[kCh];  // f16 x[16 c .. 16 c + 7], x[16 c + 8 .. 16 c + 15]
  __shared__ float xinv[kCh];           // 2^-s of chunk c
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int nw = gridDim.x * kWarps;
  auto load = [&](int r, uint4 (&a)[kU], uint4 (&b)[kU]) {
    const uint4* g4 = reinterpret_cast<const uint4*>(gc + (size_t)r * KC);
    const uint4* u4 = reinterpret_cast<const uint4*>(uc + (size_t)r * KC);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      a[u] = __ldcs(g4 + 32 * u + lane);
      b[u] = __ldcs(u4 + 32 * u + lane);
    }
  };
  uint4 ga[kU], ua[kU], gb[kU], ub[kU];  // two pairs in flight
  pdl_allow_next_grid();
  if (gw < n) load(gw, ga, ua);  // weights do not depend on the producer of x
  if (gw + nw < n) load(gw + nw, gb, ub);
  pdl_wait_prior_grid();

  {  // coherent loads: the previous kernel wrote x
    const uint4* x4 = reinterpret_cast<const uint4*>(x);
    for (int c = threadIdx.x; c < kCh; c += kWarps * 32) {
      const uint4 va = __ldcg(x4 + 2 * c), vb = __ldcg(x4 + 2 * c + 1);
      const uint32_t w[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
      float mx = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        mx = fmaxf(mx, fmaxf(fabsf(bf16_bits_to_f32(w[e] & 0xFFFFu)),
                             fabsf(bf16_bits_to_f32(w[e] >> 16))));
      const int sb = mx > 0.f ? min(f16_prescale_exponent(mx), 127) : 0;
      const float two_s = scalbnf(1.0f, sb);
      uint32_t o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        o[e] = pack_f16x2_scaled(bf16_bits_to_f32(w[e] & 0xFFFFu), bf16_bits_to_f32(w[e] >> 16), two_s);
      xlo[c] = make_uint4(o[0], o[1], o[2], o[3]);
      xhi[c] = make_uint4(o[4], o[5], o[6], o[7]);
      xinv[c] = scalbnf(1.0f, -sb);  // exact
    }
  }
  __syncthreads();
  // sum over the lane's chunks of codes . x (each chunk scaled by its 2^-s)
  auto dot = [&](const uint4 (&cw)[kU]) {
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int c = 32 * u + lane;
      const uint4 xa = xlo[c], xb = xhi[c];
      float a0 = 0.f, a1 = 0.f;
      uint32_t h0, h1;
      e4m3x4_to_f16x2(cw[u].x, h0, h1);
      fma_f16x2_f32(a0, a1, h0, xa.x);
      fma_f16x2_f32(a0, a1, h1, xa.y);
      e4m3x4_to_f16x2(cw[u].y, h0, h1);
      fma_f16x2_f32(a0, a1, h0, xa.z);
      fma_f16x2_f32(a0, a1, h1, xa.w);
      e4m3x4_to_f16x2(cw[u].z, h0, h1);
      fma_f16x2_f32(a0, a1, h0, xb.x);
      fma_f16x2_f32(a0, a1, h1, xb.y);
      e4m3x4_to_f16x2(cw[u].w, h0, h1);
      fma_f16x2_f32(a0, a1, h0, xb.z);
      fma_f16x2_f32(a0, a1, h1, xb.w);
      acc = fmaf(a0 + a1, xinv[c], acc);
    }
    return acc;
  };
  auto pair = [&](int r, const uint4 (&cg)[kU], const uint4 (&cu)[kU]) {
    const float v = warp_sum2(dot(cg), dot(cu), lane);  // lanes 0-15: gate, 16-31: up
    const float vu = __shfl_sync(0xffffffffu, v, 16);
    if (lane == 0) h[r] = f32_to_bf16_rne(silu_mul(v * gs[r], vu * us[r]));
  };
  for (int r = gw; r < n; r += 2 * nw) {  // warp-uniform
    pair(r, ga, ua);
    if (r + 2 * nw < n) load(r + 2 * nw, ga, ua);
    if (r + nw < n) {
      pair(r + nw, gb, ub);
      if (r + 3 * nw < n) load(r + 3 * nw, gb, ub);
    }
  }
}

template <int KC>
cudaError_t run_swiglu_k(const DeviceInfo& di, const uint8_t* gc, const float* gs,
                         const uint8_t* uc, const float* us, int n, const uint16_t* x,
                         uint16_t* h, cudaStream_t s, bool pdl) {
  int grid = 2 * di.sms;
  const int need = (n + kWarps - 1) / kWarps;
  if (grid > need) grid = need;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fp8_swiglu_k_kernel<KC>, gc, gs, uc, us, n, x, h);
}

template <bool SWIGLU>
cudaError_t run_fp8(const uint8_t* wa, const float* sa, const uint8_t* wb, const float* sb, int n,
                    int k, const uint16_t* x, int m, uint16_t* y, cudaStream_t s, bool pdl) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorNoDevice;
  if (m == 1) return run_pair<1, SWIGLU>(*di, wa, sa, wb, sb, n, k, x, m, y, s, pdl);
  if (m == 2) return run_pair<2, SWIGLU>(*di, wa, sa, wb, sb, n, k, x, m, y, s, pdl);
  if (m <= 4) return run_pair<4, SWIGLU>(*di, wa, sa, wb, sb, n, k, x, m, y, s, pdl);
  return run_pair<8, SWIGLU>(*di, wa, sa, wb, sb, n, k, x, m, y, s, pdl);
}

}  // namespace

cudaError_t launch_quantize_fp8(const float* w, int64_t n, int64_t k, uint8_t* codes,
                                float* scales, int32_t* status, cudaStream_t s) {
  const int64_t blocks = (n + kQThreads / 32 - 1) / (kQThreads / 32);
  quantize_fp8_kernel<<<dim3(unsigned(blocks)), kQThreads, 0, s>>>(w, n, k, codes, scales, status);
  return cudaGetLastError();
}

cudaError_t launch_fp8_matvec(const uint8_t* codes, const float* scales, int n, int k,
                              const uint16_t* x, int m, uint16_t* y, cudaStream_t s, bool pdl) {
  return run_fp8<false>(codes, scales, codes, scales, n, k, x, m, y, s, pdl);
}

cudaError_t launch_fp8_swiglu(const uint8_t* gc, const float* gs, const uint8_t* uc,
                              const float* us, int n, int k, const uint16_t* x, int m,
                              uint16_t* h, cudaStream_t s, bool pdl) {
  if (m == 1 && k == 2048) {  // SmolLM3-3B's gate/up: a warp per row pair
    const DeviceInfo* di = device_info();
    if (!di) return cudaErrorNoDevice;
    return run_swiglu_k<2048>(*di, gc, gs, uc, us, n, x, h, s, pdl);
  }
  return run_fp8<true>(gc, gs, uc, us, n, k, x, m, h, s, pdl);
}

}  // namespace tt
