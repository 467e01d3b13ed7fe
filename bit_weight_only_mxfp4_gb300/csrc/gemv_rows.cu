// Single-matrix matvecs for the down projection of a dense decode MLP:
// MXFP4 (canonical codes + E8M0 scales + optional fp32 row postscale) and
// bf16.
//
// Method: ThinTensor devlog (kerbin.cskartikey.dev/@satvikhardat), Dev Log #4
// "Why this was not just normal quantization": a selective profile quantises
// some projections and keeps the rest in bf16, and the MLP block is gate/up
// SwiGLU followed by the down projection; the project page
// (stardance.hackclub.com/projects/29750, 97.87 tok/s notes) runs whole
// layer stacks as captured CUDA graphs.  These kernels are the block's
// second step.  Both wait for the previous kernel (the gate/up SwiGLU that
// writes their x) only after their first weights are in flight
// (programmatic dependent launch), so a block captured as gate/up -> down
// streams the down weights during the gate/up kernel's tail.
//
// Layout of the work: ks warps per output row (a down projection has few,
// long rows: its K is split so that every warp of the grid has work), rows
// strided over the grid, the slices' sums added in shared memory in slice
// order; plain 128-bit loads, U 16-byte chunks per lane per step, with the
// steps double-buffered in registers so that one step's loads are in flight
// while the previous one is computed (weights are read once, evict-first);
// x is staged once per CTA in shared memory.
//  * MXFP4: lane l owns the 32-blocks l, l+32, ... of the row (one 16-byte
//    code chunk and one scale byte each); x is stored as f16, each 32-block
//    of each batch row prescaled by its own exact power of two (block max
//    -> [2^14, 2^15)), chunk-major so a warp reads 32 consecutive 16-byte
//    words.  A block's 32 products (cvt.rn.f16x2.e2m1x2, fma.rn.f32.f16,
//    exact products) are summed in fp32 and scaled once by the E8M0 factor
//    times 2^-s; the row's lanes meet in a shuffle reduction.
//  * bf16: fma.rn.f32.bf16 (exact products), x read through L1.
#include "common.cuh"
#include "launch.h"
#include "mxfp4_core.cuh"

namespace tt {
namespace {

constexpr int kWarps = 8;
constexpr int kU = 8;  // 16-byte chunks per lane in flight per row
constexpr int kRowsKMaxWarps = 16;  // one-wave MXFP4 kernel: warps per CTA at most

// The K split: a CTA's 8 warps take R = 8 / ks rows at a time, ks warps per
// row, warp (lr, sl) the sl-th slice of row rb + lr's K; the slices' sums
// meet in shared memory and are added in slice order.
struct Split {
  int ks, R, lr, sl;
  __device__ Split(int ks_, int warp) : ks(ks_), R(kWarps / ks_), lr(warp / ks_), sl(warp % ks_) {}
};

template <int MT>
__global__ void __launch_bounds__(kWarps * 32, 2)
    mxfp4_rows_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                      const float* __restrict__ post, int n, int k,
                      const uint16_t* __restrict__ x, int m, uint16_t* __restrict__ y, int ks) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float red[kWarps][MT];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Split P(ks, warp);
  const int nblk = k >> 5;
  const int bs = (nblk + ks - 1) / ks;  // blocks per slice
  const int bbeg = P.sl * bs, bend = min(nblk, bbeg + bs);
  uint4* xs = reinterpret_cast<uint4*>(smem);  // [MT][4 chunks][nblk] f16
  float* xinv = reinterpret_cast<float*>(xs + (size_t)MT * 4 * nblk);  // [MT][nblk]
  const int rstep = gridDim.x * P.R;
  const uint64_t pol = l2_evict_first_policy();

  auto load = [&](int r, int b0, uint4 (&cv)[kU], uint32_t (&sv)[kU]) {
    const uint8_t* cr = codes + (size_t)r * (k >> 1);
    const uint8_t* sr = scales + (size_t)r * nblk;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int b = b0 + 32 * u + lane;
      cv[u] = make_uint4(0u, 0u, 0u, 0u);
      sv[u] = 0u;
      if (r < n && b < bend) {
        cv[u] = ld_global_v4_hint(cr + 16 * b, pol);
        sv[u] = __ldcs(sr + b);
      }
    }
  };
  pdl_allow_next_grid();
  uint4 cv[kU], cw[kU];
  uint32_t sv[kU], sw[kU];
  load(blockIdx.x * P.R + P.lr, bbeg, cv, sv);  // weights do not depend on the previous kernel
  pdl_wait_prior_grid();

  // x: per (batch row, 32-block) exact prescale, four threads per block;
  // four chunks per thread requested at once
  const int nch = MT * (k >> 3);
  for (int c0 = 0; c0 < nch; c0 += 4 * kWarps * 32) {  // uniform trip count
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * kWarps * 32 + threadIdx.x;
      const int i = c / (k >> 3), cc = c - i * (k >> 3);
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (c < nch && i < m) v[u] = __ldcg(reinterpret_cast<const uint4*>(x + (size_t)i * k + 8 * cc));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * kWarps * 32 + threadIdx.x;
      const int i = c / (k >> 3), cc = c - i * (k >> 3);
      const uint4 w4 = v[u];
      float mx = fmaxf(fmaxf(fmaxf(fabsf(bf16_bits_to_f32(w4.x & 0xFFFFu)), fabsf(bf16_bits_to_f32(w4.x >> 16))),
                             fmaxf(fabsf(bf16_bits_to_f32(w4.y & 0xFFFFu)), fabsf(bf16_bits_to_f32(w4.y >> 16)))),
                       fmaxf(fmaxf(fabsf(bf16_bits_to_f32(w4.z & 0xFFFFu)), fabsf(bf16_bits_to_f32(w4.z >> 16))),
                             fmaxf(fabsf(bf16_bits_to_f32(w4.w & 0xFFFFu)), fabsf(bf16_bits_to_f32(w4.w >> 16)))));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (c < nch) {
        const int sb = min(f16_prescale_exponent(mx), 127);
        const float two_s = scalbnf(1.0f, sb);
        uint4 o;
        o.x = pack_f16x2_scaled(bf16_bits_to_f32(w4.x & 0xFFFFu), bf16_bits_to_f32(w4.x >> 16), two_s);
        o.y = pack_f16x2_scaled(bf16_bits_to_f32(w4.y & 0xFFFFu), bf16_bits_to_f32(w4.y >> 16), two_s);
        o.z = pack_f16x2_scaled(bf16_bits_to_f32(w4.z & 0xFFFFu), bf16_bits_to_f32(w4.z >> 16), two_s);
        o.w = pack_f16x2_scaled(bf16_bits_to_f32(w4.w & 0xFFFFu), bf16_bits_to_f32(w4.w >> 16), two_s);
        xs[((size_t)i * 4 + (cc & 3)) * nblk + (cc >> 2)] = o;  // chunk q of block b
        if ((cc & 3) == 0) xinv[(size_t)i * nblk + (cc >> 2)] = scalbnf(1.0f, -sb);  // exact
      }
    }
  }
  __syncthreads();

  auto compute = [&](float (&acc)[MT], const uint4 (&c)[kU], const uint32_t (&sc8)[kU], int b0) {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int b = b0 + 32 * u + lane;
      if (b < bend) {
        uint32_t hc[16];
        decode32(c[u], hc);
        const float sc = e8m0_to_f32(sc8[u]);
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          if (i < m) {
            uint32_t xv[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 t = xs[((size_t)i * 4 + q) * nblk + b];
              xv[4 * q + 0] = t.x;
              xv[4 * q + 1] = t.y;
              xv[4 * q + 2] = t.z;
              xv[4 * q + 3] = t.w;
            }
            acc[i] = fmaf(dot32_decoded(hc, xv), sc * xinv[(size_t)i * nblk + b], acc[i]);
          }
        }
      }
    }
  };
  // One step = kU blocks per lane, double-buffered in registers: the next
  // step's (or the next row's first step's) loads are issued before the
  // current step is computed.
  constexpr int kStep = 32 * kU;
  for (int rb = blockIdx.x * P.R; rb < n; rb += rstep) {  // uniform over the CTA
    const int r = rb + P.lr;
    float acc[MT];
#pragma unroll
    for (int i = 0; i < MT; ++i) acc[i] = 0.f;
    for (int b0 = bbeg;; b0 += 2 * kStep) {
      const bool has_w = b0 + kStep < bend;
      if (has_w) load(r, b0 + kStep, cw, sw);
      if (r < n) compute(acc, cv, sv, b0);
      const bool more = b0 + 2 * kStep < bend;
      if (more) load(r, b0 + 2 * kStep, cv, sv);
      else load(r + rstep, bbeg, cv, sv);  // the next row in flight during the rest
      if (has_w && r < n) compute(acc, cw, sw, b0 + kStep);
      if (!more) break;
    }
    if (P.ks == 1) {  // whole rows per warp: no exchange
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const float v = warp_sum(acc[i]);
        if (lane == 0 && r < n && i < m)
          y[(size_t)i * n + r] = f32_to_bf16_rne(v * (post ? post[r] : 1.f));
      }
      continue;
    }
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      const float v = warp_sum(acc[i]);
      if (lane == 0) red[warp][i] = v;
    }
    __syncthreads();
    if (threadIdx.x < P.R * MT) {
      const int lr = threadIdx.x / MT, i = threadIdx.x - lr * MT;
      const int rr = rb + lr;
      if (rr < n && i < m) {
        float v = 0.f;
        for (int s2 = 0; s2 < P.ks; ++s2) v += red[lr * P.ks + s2][i];
        y[(size_t)i * n + rr] = f32_to_bf16_rne(v * (post ? post[rr] : 1.f));
      }
    }
    __syncthreads();
  }
}

// m = 1 with K fixed at compile time (the down projection of the models the
// library serves): one CTA per SM of ceil(n / SMs) warps (at most
// kRowsKMaxWarps), so the rows spread evenly over the SMs and each SM stages
// x once; a warp owns whole rows, and all of a row's code chunks
// and scale bytes (U = ceil(K / 1024) per lane) are requested in one wave,
// the first row's before the dependency wait, so that the whole matrix is
// in flight while the previous kernel finishes.  Only the one partial chunk
// of a lane is tested against the row's end; every offset is an immediate.
// Same arithmetic as mxfp4_rows_kernel at m = 1 (measured there: a fixed
// 8-chunk step that leaves two thirds of the second step empty at
// K = 11008, and 6.3 instructions per weight).
template <int KC>
__global__ void __launch_bounds__(kRowsKMaxWarps * 32, 1)
    mxfp4_rows_k_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                        const float* __restrict__ post, int n, int /*k*/,
                        const uint16_t* __restrict__ x, int /*m*/, uint16_t* __restrict__ y,
                        int /*ks*/) {
  static_assert(KC % 32 == 0 && KC / 32 <= 32 * 12, "one wave of at most 12 chunks per lane");
  constexpr int kNblk = KC / 32;
  constexpr int kU1 = (kNblk + 31) / 32;  // chunks per lane
  constexpr int kFull = kNblk / 32;       // chunks every lane has
  constexpr int kCh = KC / 8;             // 16-byte chunks of x
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int W = blockDim.x >> 5;  // warps of the CTA
  uint4* xs = reinterpret_cast<uint4*>(smem);              // [4 chunks][nblk] f16
  float* xinv = reinterpret_cast<float*>(xs + 4 * kNblk);  // [nblk]
  const uint64_t pol = l2_evict_first_policy();
  const int rstep = gridDim.x * W;

  uint4 cv[kU1];
  uint32_t sv[kU1];
  auto load = [&](int r) {
    const uint8_t* cr = codes + (size_t)r * (KC / 2);
    const uint8_t* sr = scales + (size_t)r * kNblk;
#pragma unroll
    for (int u = 0; u < kU1; ++u) {
      const int b = 32 * u + lane;
      cv[u] = make_uint4(0u, 0u, 0u, 0u);
      sv[u] = 0u;
      if (u < kFull || b < kNblk) {
        cv[u] = ld_global_v4_hint(cr + 16 * b, pol);
        sv[u] = __ldcs(sr + b);
      }
    }
  };
  int r = blockIdx.x * W + warp;  // warp-uniform
  pdl_allow_next_grid();
  if (r < n) load(r);  // weights do not depend on the previous kernel
  pdl_wait_prior_grid();

  // x: per 32-block exact prescale, four threads per block (as above)
  for (int c0 = 0; c0 < kCh; c0 += 4 * (int)blockDim.x) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * (int)blockDim.x + threadIdx.x;
      v[u] = c < kCh ? __ldcg(reinterpret_cast<const uint4*>(x) + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * (int)blockDim.x + threadIdx.x;
      const uint4 w4 = v[u];
      float mx = fmaxf(fmaxf(fmaxf(fabsf(bf16_bits_to_f32(w4.x & 0xFFFFu)), fabsf(bf16_bits_to_f32(w4.x >> 16))),
                             fmaxf(fabsf(bf16_bits_to_f32(w4.y & 0xFFFFu)), fabsf(bf16_bits_to_f32(w4.y >> 16)))),
                       fmaxf(fmaxf(fabsf(bf16_bits_to_f32(w4.z & 0xFFFFu)), fabsf(bf16_bits_to_f32(w4.z >> 16))),
                             fmaxf(fabsf(bf16_bits_to_f32(w4.w & 0xFFFFu)), fabsf(bf16_bits_to_f32(w4.w >> 16)))));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (c < kCh) {
        const int sb = min(f16_prescale_exponent(mx), 127);
        const float two_s = scalbnf(1.0f, sb);
        uint4 o;
        o.x = pack_f16x2_scaled(bf16_bits_to_f32(w4.x & 0xFFFFu), bf16_bits_to_f32(w4.x >> 16), two_s);
        o.y = pack_f16x2_scaled(bf16_bits_to_f32(w4.y & 0xFFFFu), bf16_bits_to_f32(w4.y >> 16), two_s);
        o.z = pack_f16x2_scaled(bf16_bits_to_f32(w4.z & 0xFFFFu), bf16_bits_to_f32(w4.z >> 16), two_s);
        o.w = pack_f16x2_scaled(bf16_bits_to_f32(w4.w & 0xFFFFu), bf16_bits_to_f32(w4.w >> 16), two_s);
        xs[(c & 3) * kNblk + (c >> 2)] = o;  // chunk q of block b
        if ((c & 3) == 0) xinv[c >> 2] = scalbnf(1.0f, -sb);  // exact
      }
    }
  }
  __syncthreads();

  for (; r < n; r += rstep) {
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < kU1; ++u) {
      const int b = 32 * u + lane;
      if (u < kFull || b < kNblk) {
        uint32_t hc[16], xv[16];
        decode32(cv[u], hc);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 t = xs[q * kNblk + b];
          xv[4 * q + 0] = t.x;
          xv[4 * q + 1] = t.y;
          xv[4 * q + 2] = t.z;
          xv[4 * q + 3] = t.w;
        }
        acc = fmaf(dot32_decoded(hc, xv), e8m0_to_f32(sv[u]) * xinv[b], acc);
      }
    }
    if (r + rstep < n) load(r + rstep);  // the warp's next row, in flight during the reduction
    const float v = warp_sum(acc);
    if (lane == 0) y[r] = f32_to_bf16_rne(v * (post ? post[r] : 1.f));
  }
}

template <int MT>
__global__ void __launch_bounds__(kWarps * 32, 2)
    bf16_rows_kernel(const uint16_t* __restrict__ w, int n, int k,
                     const uint16_t* __restrict__ x, int m, uint16_t* __restrict__ y, int ks) {
  __shared__ float red[kWarps][MT];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Split P(ks, warp);
  const int cpr = k >> 3;  // 16-byte chunks per row
  const int cs = (cpr + ks - 1) / ks;
  const int cbeg = P.sl * cs, cend = min(cpr, cbeg + cs);
  const int rstep = gridDim.x * P.R;
  const uint4* x4 = reinterpret_cast<const uint4*>(x);
  auto load = [&](int r, int c0, uint4 (&wv)[kU]) {
    const uint4* w4 = reinterpret_cast<const uint4*>(w + (size_t)r * k);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int c = c0 + u * 32 + lane;
      wv[u] = (r < n && c < cend) ? __ldcs(w4 + c) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  pdl_allow_next_grid();
  uint4 wv[kU], ww[kU];
  load(blockIdx.x * P.R + P.lr, cbeg, wv);  // weights do not depend on the previous kernel
  pdl_wait_prior_grid();
  auto compute = [&](float (&a0)[MT], float (&a1)[MT], const uint4 (&wc)[kU], int c0) {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int c = c0 + u * 32 + lane;
      if (c < cend) {
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          if (i < m) {
            const uint4 xv = __ldca(x4 + (size_t)i * cpr + c);
            fma_bf16x2_f32(a0[i], a1[i], wc[u].x, xv.x);
            fma_bf16x2_f32(a0[i], a1[i], wc[u].y, xv.y);
            fma_bf16x2_f32(a0[i], a1[i], wc[u].z, xv.z);
            fma_bf16x2_f32(a0[i], a1[i], wc[u].w, xv.w);
          }
        }
      }
    }
  };
  constexpr int kStep = 32 * kU;
  for (int rb = blockIdx.x * P.R; rb < n; rb += rstep) {  // uniform over the CTA
    const int r = rb + P.lr;
    float a0[MT], a1[MT];
#pragma unroll
    for (int i = 0; i < MT; ++i) a0[i] = a1[i] = 0.f;
    for (int c0 = cbeg;; c0 += 2 * kStep) {  // double-buffered steps, as above
      const bool has_w = c0 + kStep < cend;
      if (has_w) load(r, c0 + kStep, ww);
      if (r < n) compute(a0, a1, wv, c0);
      const bool more = c0 + 2 * kStep < cend;
      if (more) load(r, c0 + 2 * kStep, wv);
      else load(r + rstep, cbeg, wv);
      if (has_w && r < n) compute(a0, a1, ww, c0 + kStep);
      if (!more) break;
    }
    if (P.ks == 1) {  // whole rows per warp: no exchange
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const float v = warp_sum(a0[i] + a1[i]);
        if (lane == 0 && r < n && i < m) y[(size_t)i * n + r] = f32_to_bf16_rne(v);
      }
      continue;
    }
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      const float v = warp_sum(a0[i] + a1[i]);
      if (lane == 0) red[warp][i] = v;
    }
    __syncthreads();
    if (threadIdx.x < P.R * MT) {
      const int lr = threadIdx.x / MT, i = threadIdx.x - lr * MT;
      const int rr = rb + lr;
      if (rr < n && i < m) {
        float v = 0.f;
        for (int s2 = 0; s2 < P.ks; ++s2) v += red[lr * P.ks + s2][i];
        y[(size_t)i * n + rr] = f32_to_bf16_rne(v);
      }
    }
    __syncthreads();
  }
}

// Warps per row: enough (row, slice) work items for every warp of a full
// grid several times over (long rows with few outputs, as in a down
// projection, are split), while a slice keeps at least 4 KB of a row.
int choose_split(const DeviceInfo& di, int n, int64_t row_bytes) {
  int ks = 1;
  while (ks < kWarps && (int64_t)n * ks < (int64_t)2 * 2 * di.sms * kWarps &&
         row_bytes / (2 * ks) >= 4096)
    ks *= 2;
  return ks;
}

template <class Kern, class... Args>
cudaError_t launch_rows(const DeviceInfo& di, Kern kern, int n, int ks, int smem, cudaStream_t s,
                        bool pdl, Args... args) {
  if (smem > di.smem_optin) return cudaErrorInvalidConfiguration;
  if (smem > 0) {
    const cudaError_t e = ensure_smem(di, kern, smem);
    if (e != cudaSuccess) return e;
  }
  const int R = kWarps / ks;
  int grid = 2 * di.sms;
  const int need = (n + R - 1) / R;
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
  return cudaLaunchKernelEx(&cfg, kern, args..., ks);
}

// One CTA per SM with ceil(n / SMs) warps (rows spread evenly over the SMs).
template <class Kern, class... Args>
cudaError_t launch_rows_k(const DeviceInfo& di, Kern kern, int n, int smem, cudaStream_t s,
                          bool pdl, Args... args) {
  if (smem > di.smem_optin) return cudaErrorInvalidConfiguration;
  const cudaError_t e = ensure_smem(di, kern, smem);
  if (e != cudaSuccess) return e;
  int warps = (n + di.sms - 1) / di.sms;
  if (warps > kRowsKMaxWarps) warps = kRowsKMaxWarps;
  if (warps < 1) warps = 1;
  int grid = (n + warps - 1) / warps;
  if (grid > di.sms) grid = di.sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(warps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args..., 1);
}

template <int MT>
cudaError_t run_mxfp4_rows(const DeviceInfo& di, const uint8_t* codes, const uint8_t* scales,
                           const float* post, int n, int k, const uint16_t* x, int m, uint16_t* y,
                           cudaStream_t s, bool pdl) {
  const int smem = MT * (2 * k + 4 * (k / 32));
  return launch_rows(di, mxfp4_rows_kernel<MT>, n, choose_split(di, n, k / 2 + k / 32), smem, s,
                     pdl, codes, scales, post, n, k, x, m, y);
}

// bf16 at m = 1 with K fixed at compile time (the down projection of the
// models the library serves): the CTA's 8 warps split one row (a slice of
// K each, U = ceil(K / 2048) 16-byte chunks per lane, all requested at
// once); rows go round-robin over the grid, the slices of the CTA's next
// rows are requested while the current one is computed, and the slices'
// sums meet in shared memory in slice order.  One row per CTA step keeps the rows of a
// call even over the CTAs (2048 rows: 7 steps on the busiest CTA against
// 6.7 on average, where 2 rows per step leave 4 against 3.4).
// Rows of a CTA in flight (measured at K = 11008, N = 2048: 9.98 / 9.47 /
// 8.96 us for 1 / 2 / 3; 3 uses 114 registers, so two CTAs still fit an SM).
#ifndef TT_BF16K_DEPTH
#define TT_BF16K_DEPTH 3
#endif
template <int KC>
__global__ void __launch_bounds__(kWarps * 32, 2)
    bf16_rows_k_kernel(const uint16_t* __restrict__ w, int n, int /*k*/,
                       const uint16_t* __restrict__ x, int /*m*/, uint16_t* __restrict__ y,
                       int /*ks*/) {
  static_assert(KC % (8 * kWarps) == 0, "whole chunks per slice");
  constexpr int kCpr = KC / 8;            // 16-byte chunks per row
  constexpr int kCps = kCpr / kWarps;     // per slice
  constexpr int kU1 = (kCps + 31) / 32;   // per lane
  constexpr int kFull = kCps / 32;        // chunks every lane has
  __shared__ float red[2][kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = warp * kCps;
  const uint4* x4 = reinterpret_cast<const uint4*>(x);
  auto load = [&](int r, uint4 (&wv)[kU1]) {
    const uint4* w4 = reinterpret_cast<const uint4*>(w + (size_t)r * KC) + c0;
#pragma unroll
    for (int u = 0; u < kU1; ++u) {
      const int c = 32 * u + lane;
      wv[u] = (u < kFull || c < kCps) ? __ldcs(w4 + c) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  auto row = [&](int r, const uint4 (&wv)[kU1], int buf) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int u = 0; u < kU1; ++u) {
      const int c = 32 * u + lane;
      if (u < kFull || c < kCps) {
        const uint4 xv = __ldca(x4 + c0 + c);
        fma_bf16x2_f32(a0, a1, wv[u].x, xv.x);
        fma_bf16x2_f32(a0, a1, wv[u].y, xv.y);
        fma_bf16x2_f32(a0, a1, wv[u].z, xv.z);
        fma_bf16x2_f32(a0, a1, wv[u].w, xv.w);
      }
    }
    const float v = warp_sum(a0 + a1);
    if (lane == 0) red[buf][warp] = v;
    __syncthreads();  // red[buf] of this row is complete; red[buf ^ 1] is free
    if (threadIdx.x == 0) {
      float t = 0.f;
#pragma unroll
      for (int sl = 0; sl < kWarps; ++sl) t += red[buf][sl];
      y[r] = f32_to_bf16_rne(t);
    }
  };
  constexpr int D = TT_BF16K_DEPTH;  // rows of this CTA in flight
  const int G = gridDim.x;
  uint4 wbuf[D][kU1];
  pdl_allow_next_grid();
#pragma unroll
  for (int d = 0; d < D; ++d)  // weights do not depend on the previous kernel
    if ((int)blockIdx.x + d * G < n) load(blockIdx.x + d * G, wbuf[d]);
  pdl_wait_prior_grid();
  int q = 0;  // rows done: alternates the reduction buffer
  for (int r = blockIdx.x; r < n; r += D * G) {  // uniform over the CTA
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const int rr = r + d * G;
      if (rr < n) {
        row(rr, wbuf[d], q & 1);
        ++q;
        if (rr + D * G < n) load(rr + D * G, wbuf[d]);  // this buffer's next row
      }
    }
  }
}

}  // namespace

cudaError_t launch_mxfp4_rows(const uint8_t* codes, const uint8_t* scales, const float* post,
                              int n, int k, const uint16_t* x, int m, uint16_t* y, cudaStream_t s,
                              bool pdl) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorNoDevice;
  // SmolLM3-3B's down projection (K = 11008) gets the one-wave kernel
  if (m == 1 && k == 11008)
    return launch_rows_k(*di, mxfp4_rows_k_kernel<11008>, n, 2 * k + 4 * (k / 32), s, pdl, codes,
                         scales, post, n, k, x, m, y);
  if (m == 1) return run_mxfp4_rows<1>(*di, codes, scales, post, n, k, x, m, y, s, pdl);
  if (m == 2) return run_mxfp4_rows<2>(*di, codes, scales, post, n, k, x, m, y, s, pdl);
  if (m <= 4) return run_mxfp4_rows<4>(*di, codes, scales, post, n, k, x, m, y, s, pdl);
  return run_mxfp4_rows<8>(*di, codes, scales, post, n, k, x, m, y, s, pdl);
}

cudaError_t launch_bf16_rows(const uint16_t* w, int n, int k, const uint16_t* x, int m,
                             uint16_t* y, cudaStream_t s, bool pdl) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorNoDevice;
  // SmolLM3-3B's down projection (K = 11008): one row per CTA step
  if (m == 1 && k == 11008)
    return launch_rows(*di, bf16_rows_k_kernel<11008>, n, kWarps, 0, s, pdl, w, n, k, x, m, y);
  const int ks = choose_split(*di, n, int64_t(2) * k);
  if (m == 1) return launch_rows(*di, bf16_rows_kernel<1>, n, ks, 0, s, pdl, w, n, k, x, m, y);
  if (m == 2) return launch_rows(*di, bf16_rows_kernel<2>, n, ks, 0, s, pdl, w, n, k, x, m, y);
  if (m <= 4) return launch_rows(*di, bf16_rows_kernel<4>, n, ks, 0, s, pdl, w, n, k, x, m, y);
  return launch_rows(*di, bf16_rows_kernel<8>, n, ks, 0, s, pdl, w, n, k, x, m, y);
}

}  // namespace tt
