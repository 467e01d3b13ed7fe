// Grouped affine INT4 matvec for the dense Q/K/V/O projections, m = 1..8.
//
// Method: the ThinTensor project page (stardance.hackclub.com/projects/29750)
// runs Q/K/V/O as INT4 under dense_int4_layers="all" (97.87 tok/s notes), with
// affine groups whose last group may be partial (fixes list).  Per row and
// group g: w = (q - zp_g) * s_g, so
//     y = sum_g s_g * sum_{k in g} (q_k - zp_g) * x_k.
//
// Kernel: one warp per output row; lane l owns the 32-weight chunks l, l+32,
// ... of the row (group % 32 == 0, so a chunk never straddles two groups).
// A chunk's 16 code bytes arrive with one 128-bit load.  Nibble pairs
// (q_i, q_{i+4}) of each 32-bit word become f16x2 (1024 + q) with one LOP3
// against the exponent pattern 0x6400, and one HSUB2 of (1024 + zp) turns
// them into the exact small integers q - zp; the products with x (f16 after
// an exact power-of-two prescale per 32-chunk, stored in shared memory in the
// same pair order) accumulate in fp32 with fma.rn.f32.f16, and each chunk's
// sum is scaled by its group's fp16 scale times the chunk's inverse
// prescale.  A warp requests its rows' codes, scales and zero points before
// the dependency wait on the previous kernel.
#include "common.cuh"
#include "launch.h"
#include "mxfp4_core.cuh"

namespace tt {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t bits) {
  uint32_t d;
  // d = (a & mask) | bits
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));
  return d;
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&b);
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Sum over one 32-weight chunk of (q - zp) * x, x given as 16 f16x2 values
// in the pair order (x[8t+i], x[8t+i+4]) for word t, pair i.
__device__ __forceinline__ float chunk_dot(const uint4& c, uint32_t zz, const uint32_t* xv) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t p0 = hsub2(lop3_and_or(w[t], 0x000F000Fu, 0x64006400u), zz);
    const uint32_t p1 = hsub2(lop3_and_or(w[t] >> 4, 0x000F000Fu, 0x64006400u), zz);
    const uint32_t p2 = hsub2(lop3_and_or(w[t] >> 8, 0x000F000Fu, 0x64006400u), zz);
    const uint32_t p3 = hsub2(lop3_and_or(w[t] >> 12, 0x000F000Fu, 0x64006400u), zz);
    fma_f16x2_f32(a0, a1, p0, xv[4 * t + 0]);
    fma_f16x2_f32(a2, a3, p1, xv[4 * t + 1]);
    fma_f16x2_f32(a0, a1, p2, xv[4 * t + 2]);
    fma_f16x2_f32(a2, a3, p3, xv[4 * t + 3]);
  }
  return (a0 + a1) + (a2 + a3);
}

// RPW rows per warp and pass: all of a pass's codes, scales and zero points
// are requested before the dependency wait (the first pass) or before the
// previous pass is reduced (the others), so only the x staging and the math
// follow the wait.
template <int CPL, int MT, int RPW>
__global__ void __launch_bounds__(kThreads, 2)
    int4_matvec_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                       const uint8_t* __restrict__ zp, int n, int k, int group,
                       const uint16_t* __restrict__ x, int m, uint16_t* __restrict__ y) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = k >> 5;                     // 32-weight chunks per row
  const int ng = (k + group - 1) / group;     // groups per row
  const int zb = (ng + 1) >> 1;               // zero-point bytes per row
  const int gw = blockIdx.x * kWarps + warp;
  const int nw = gridDim.x * kWarps;
  uint4* xs = reinterpret_cast<uint4*>(smem);                          // [MT][4][nch]
  float* xinv = reinterpret_cast<float*>(xs + (size_t)MT * 4 * nch);  // [MT][nch]

  pdl_allow_next_grid();

  // This warp's rows of one pass (row r + u * nw): codes, and per chunk the
  // group's scale and f16x2 (1024 + zp).  None depends on the previous kernel.
  // Wide rows (many chunks per lane) take their scales in the math loop
  // instead, to stay within the registers.
  constexpr bool kPre = CPL * RPW <= 12;
  uint4 cw[RPW][CPL];
  float sc[RPW][CPL];
  uint32_t zz[RPW][CPL];
  auto scale_of = [&](int row, int j) {
    return row < n && j < nch
               ? __half2float(__ushort_as_half(__ldg(scales + (size_t)row * ng + (j * 32) / group)))
               : 0.f;
  };
  auto zz_of = [&](int row, int j) {
    const int g = (j * 32) / group;
    const uint32_t z =
        row < n && j < nch ? (__ldg(zp + (size_t)row * zb + (g >> 1)) >> (4 * (g & 1))) & 15u : 0u;
    return 0x64006400u + z * 0x00010001u;
  };
  auto load_rows = [&](int r) {
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
      const int row = r + u * nw;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int j = c * 32 + lane;
        cw[u][c] = row < n && j < nch
                       ? __ldcs(reinterpret_cast<const uint4*>(codes + (size_t)row * (k >> 1)) + j)
                       : make_uint4(0, 0, 0, 0);
        if constexpr (kPre) {
          sc[u][c] = scale_of(row, j);
          zz[u][c] = zz_of(row, j);
        }
      }
    }
  };
  load_rows(gw);
  pdl_wait_prior_grid();

  // x -> f16 in pair order, each 32-chunk of each row prescaled by its own
  // exact power of two 2^s (chunk max |x| -> [2^14, 2^15)); 2^-s is folded
  // into the chunk's group scale below.  Four threads share a chunk (8
  // values each) and meet in two shuffles.
  const int n8 = MT * (k >> 3);
  for (int c0 = 0; c0 < n8; c0 += kThreads) {  // uniform trip count
    const int c = c0 + threadIdx.x;
    const int i = c / (k >> 3), t8 = c - i * (k >> 3);  // x[8*t8 .. 8*t8+7] of row i
    uint4 v = make_uint4(0, 0, 0, 0);
    if (c < n8 && i < m) v = __ldcg(reinterpret_cast<const uint4*>(x + (size_t)i * k) + t8);
    const float e0 = bf16_bits_to_f32(v.x & 0xFFFFu), e1 = bf16_bits_to_f32(v.x >> 16);
    const float e2 = bf16_bits_to_f32(v.y & 0xFFFFu), e3 = bf16_bits_to_f32(v.y >> 16);
    const float e4 = bf16_bits_to_f32(v.z & 0xFFFFu), e5 = bf16_bits_to_f32(v.z >> 16);
    const float e6 = bf16_bits_to_f32(v.w & 0xFFFFu), e7 = bf16_bits_to_f32(v.w >> 16);
    float mx = fmaxf(fmaxf(fmaxf(fabsf(e0), fabsf(e1)), fmaxf(fabsf(e2), fabsf(e3))),
                     fmaxf(fmaxf(fabsf(e4), fabsf(e5)), fmaxf(fabsf(e6), fabsf(e7))));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (c < n8) {
      const int sb = min(f16_prescale_exponent(mx), 127);
      const float two_s = scalbnf(1.0f, sb);
      uint4 o;
      o.x = pack_f16x2_scaled(e0, e4, two_s);
      o.y = pack_f16x2_scaled(e1, e5, two_s);
      o.z = pack_f16x2_scaled(e2, e6, two_s);
      o.w = pack_f16x2_scaled(e3, e7, two_s);
      // word t = t8 % 4 of chunk j = t8 / 4
      xs[((size_t)i * 4 + (t8 & 3)) * nch + (t8 >> 2)] = o;
      if ((t8 & 3) == 0) xinv[(size_t)i * nch + (t8 >> 2)] = scalbnf(1.0f, -sb);  // exact
    }
  }
  __syncthreads();

  for (int r = gw; r < n; r += RPW * nw) {
    float acc[RPW][MT];
#pragma unroll
    for (int u = 0; u < RPW; ++u)
#pragma unroll
      for (int i = 0; i < MT; ++i) acc[u][i] = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int j = c * 32 + lane;
      if (j < nch) {
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          if (i < m) {
            uint32_t xv[16];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const uint4 q = xs[((size_t)i * 4 + t) * nch + j];
              xv[4 * t + 0] = q.x;
              xv[4 * t + 1] = q.y;
              xv[4 * t + 2] = q.z;
              xv[4 * t + 3] = q.w;
            }
            const float xi = xinv[(size_t)i * nch + j];
#pragma unroll
            for (int u = 0; u < RPW; ++u) {  // rows past n hold zero codes and scales
              const int row = r + u * nw;
              const float scv = kPre ? sc[u][c] : scale_of(row, j);
              const uint32_t zzv = kPre ? zz[u][c] : zz_of(row, j);
              acc[u][i] = fmaf(chunk_dot(cw[u][c], zzv, xv), scv * xi, acc[u][i]);
            }
          }
        }
      }
    }
    // request the next pass's rows before reducing these
    load_rows(r + RPW * nw);
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
      const int row = r + u * nw;
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const float v = warp_sum(acc[u][i]);
        if (lane == 0 && row < n && i < m) {
          __nv_bfloat16 b = __float2bfloat16_rn(v);
          y[(size_t)i * n + row] = *reinterpret_cast<uint16_t*>(&b);
        }
      }
    }
  }
}


// ---------------------------------------------------------------------------
// m = 1, group 128: the multiply-adds of a row pair on mma.sync m16n8k16
// (f16 x f16 -> fp32), in the diagonal form of the FP8 kernel.  A step
// covers 8 groups (1024 k): A row g holds 16 k of group 8t+g of the pair's
// first row and A row 8+g the same k of its second row, B column c holds x
// of group 8t+c, so over the step's 8 MMAs D[g][g] and D[8+g][g] are the two
// rows' dot products over exactly one group; the group's fp16 scale (and
// x's per-group inverse prescale) is applied to them once.  Lane (g, q)
// owns the 32 weights 32q.. of its group: one 16-byte code load per row,
// decoded as above into the exact (q - zp) f16x2 pairs that are the A
// fragments.  x is prescaled per 128-group (R16) and staged once per CTA in
// shared memory already in B-fragment order.  A warp owns one or two row
// pairs, all requested before the dependency wait, so the whole matrix is
// in flight by then, with about one CTA per SM left free for the next
// kernel's CTAs to do the same.
// ---------------------------------------------------------------------------
constexpr int kMmaCtaWarps = 8;

template <int ST, int PPW>  // steps of 1024 k (k <= 1024 * ST); row pairs per warp
__global__ void __launch_bounds__(kMmaCtaWarps * 32, 2)
    int4_mma_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                    const uint8_t* __restrict__ zp, int n, int k,
                    const uint16_t* __restrict__ x, uint16_t* __restrict__ y) {
  __shared__ uint4 xs[ST][4][32];  // step, 16-byte word, lane: B fragments
  __shared__ float xis[ST][8];     // inverse prescale of group 8t+g
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int ng = (k + 127) >> 7;  // groups per row (the last may be partial)
  const int zb = (ng + 1) >> 1;
  const int npairs = (n + 1) >> 1;
  const int gw = blockIdx.x * kMmaCtaWarps + warp, nw = gridDim.x * kMmaCtaWarps;

  uint4 c[PPW][2][ST];      // codes of the lane's piece, rows 2p and 2p + 1
  uint32_t zz[PPW][2][ST];  // f16x2 (1024 + zp) of the piece's group
  float sc[PPW][2][ST];     // the group's scale (0 past the end)
  auto load_pair = [&](int u, int p) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = 2 * p + r;
#pragma unroll
      for (int t = 0; t < ST; ++t) {
        const int grp = 8 * t + g;
        const bool ok = row < n && p < npairs && grp < ng;
        const int kk = 128 * grp + 32 * q;
        c[u][r][t] = ok && kk < k
                      ? __ldcs(reinterpret_cast<const uint4*>(codes + (size_t)row * (k >> 1) +
                                                              (kk >> 1)))
                      : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t z = ok ? (__ldg(zp + (size_t)row * zb + (grp >> 1)) >> (4 * (grp & 1))) & 15u : 0u;
        zz[u][r][t] = 0x64006400u + z * 0x00010001u;
        sc[u][r][t] = ok ? __half2float(__ushort_as_half(__ldg(scales + (size_t)row * ng + grp))) : 0.f;
      }
    }
  };
  // the warp's pairs gw + i * nw, all requested before the wait
#pragma unroll
  for (int u = 0; u < PPW; ++u) load_pair(u, gw + u * nw);
  pdl_allow_next_grid();
  pdl_wait_prior_grid();  // x comes from the preceding kernel

  // warp t stages step t of x: its lanes' pieces as f16 in the pair order
  // (x[8w+i], x[8w+i+4]), each 128-group prescaled by its exact power of two
  if (warp < ST) {
    const int t = warp;
    const int kk = 128 * (8 * t + g) + 32 * q;
    uint4 v[4];
#pragma unroll
    for (int w = 0; w < 4; ++w)
      v[w] = kk < k ? __ldcg(reinterpret_cast<const uint4*>(x + kk) + w) : make_uint4(0u, 0u, 0u, 0u);
    float e[32];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t u[4] = {v[w].x, v[w].y, v[w].z, v[w].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        e[8 * w + 2 * h] = bf16_bits_to_f32(u[h] & 0xFFFFu);
        e[8 * w + 2 * h + 1] = bf16_bits_to_f32(u[h] >> 16);
      }
    }
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(e[i]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));  // the group's 4 pieces
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const int sb = min(f16_prescale_exponent(mx), 127);
    const float two_s = scalbnf(1.0f, sb);
    if (q == 0) xis[t][g] = scalbnf(1.0f, -sb);  // exact
#pragma unroll
    for (int w = 0; w < 4; ++w)
      xs[t][w][lane] = make_uint4(pack_f16x2_scaled(e[8 * w + 0], e[8 * w + 4], two_s),
                                  pack_f16x2_scaled(e[8 * w + 1], e[8 * w + 5], two_s),
                                  pack_f16x2_scaled(e[8 * w + 2], e[8 * w + 6], two_s),
                                  pack_f16x2_scaled(e[8 * w + 3], e[8 * w + 7], two_s));
  }
  __syncthreads();

  const bool diag = q == (g >> 1);  // this lane holds D[g][g] and D[8+g][g]
#pragma unroll
  for (int u = 0; u < PPW; ++u) {
    const int p = gw + u * nw;
    if (p >= npairs) break;
    float acc[2] = {0.f, 0.f};
#pragma unroll
    for (int t = 0; t < ST; ++t) {
      uint32_t xb[16];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint4 xv = xs[t][w][lane];
        xb[4 * w] = xv.x;
        xb[4 * w + 1] = xv.y;
        xb[4 * w + 2] = xv.z;
        xb[4 * w + 3] = xv.w;
      }
      uint32_t pa[16], pb[16];
      const uint32_t wa[4] = {c[u][0][t].x, c[u][0][t].y, c[u][0][t].z, c[u][0][t].w};
      const uint32_t wb[4] = {c[u][1][t].x, c[u][1][t].y, c[u][1][t].z, c[u][1][t].w};
#pragma unroll
      for (int w = 0; w < 4; ++w)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          pa[4 * w + i] = hsub2(lop3_and_or(wa[w] >> (4 * i), 0x000F000Fu, 0x64006400u), zz[u][0][t]);
          pb[4 * w + i] = hsub2(lop3_and_or(wb[w] >> (4 * i), 0x000F000Fu, 0x64006400u), zz[u][1][t]);
        }
      float d0[4], d1[4];  // two accumulation chains
      mma_16816_z(d0, pa[0], pb[0], pa[1], pb[1], xb[0], xb[1]);
      mma_16816_z(d1, pa[2], pb[2], pa[3], pb[3], xb[2], xb[3]);
#pragma unroll
      for (int m = 2; m < 8; m += 2) {
        mma_16816(d0, pa[2 * m], pb[2 * m], pa[2 * m + 1], pb[2 * m + 1], xb[2 * m], xb[2 * m + 1]);
        mma_16816(d1, pa[2 * m + 2], pb[2 * m + 2], pa[2 * m + 3], pb[2 * m + 3], xb[2 * m + 2],
                  xb[2 * m + 3]);
      }
      if (diag) {
        const int e0 = g & 1;
        const float xi = xis[t][g];
        acc[0] = fmaf(d0[e0] + d1[e0], sc[u][0][t] * xi, acc[0]);
        acc[1] = fmaf(d0[2 + e0] + d1[2 + e0], sc[u][1][t] * xi, acc[1]);
      }
    }
    const float ya = warp_sum(acc[0]), yb = warp_sum(acc[1]);  // other lanes hold 0
    if (lane == 0) {
      y[2 * p] = f32_to_bf16_bits(ya);
      if (2 * p + 1 < n) y[2 * p + 1] = f32_to_bf16_bits(yb);
    }
  }
}

template <int CPL, int MT, int RPW>
cudaError_t run(const DeviceInfo& di, const uint8_t* codes, const uint16_t* scales,
                const uint8_t* zp, int n, int k, int group, const uint16_t* x, int m,
                uint16_t* y, cudaStream_t s, bool pdl) {
  const int smem = MT * 4 * (k >> 5) * 16 + MT * (k >> 5) * 4;
  if (smem > di.smem_optin) return cudaErrorInvalidConfiguration;
  auto kern = int4_matvec_kernel<CPL, MT, RPW>;
  cudaError_t e = ensure_smem(di, kern, smem);
  if (e != cudaSuccess) return e;
  int grid = 2 * di.sms;
  const int need = (n + kWarps * RPW - 1) / (kWarps * RPW);
  if (grid > need) grid = need;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, codes, scales, zp, n, k, group, x, m, y);
}


template <int ST, int PPW>
cudaError_t run_mma(const DeviceInfo& di, const uint8_t* codes, const uint16_t* scales,
                    const uint8_t* zp, int n, int k, const uint16_t* x, uint16_t* y,
                    cudaStream_t s, bool pdl) {
  const int npairs = (n + 1) / 2;
  const int grid = (npairs + kMmaCtaWarps * PPW - 1) / (kMmaCtaWarps * PPW);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMmaCtaWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, int4_mma_kernel<ST, PPW>, codes, scales, zp, n, k, x, y);
}

// Pairs per warp: one pass over the rows with about one CTA per SM (two
// when the rows need more), so the next kernel's CTAs can be resident
// early and request their weights before their own wait.
template <int ST>
cudaError_t run_mma_ppw(const DeviceInfo& di, const uint8_t* codes, const uint16_t* scales,
                        const uint8_t* zp, int n, int k, const uint16_t* x, uint16_t* y,
                        cudaStream_t s, bool pdl) {
  const int npairs = (n + 1) / 2;
  if (npairs <= kMmaCtaWarps * di.sms)
    return run_mma<ST, 1>(di, codes, scales, zp, n, k, x, y, s, pdl);
  return run_mma<ST, 2>(di, codes, scales, zp, n, k, x, y, s, pdl);
}

template <int CPL>
cudaError_t run_m(const DeviceInfo& di, const uint8_t* codes, const uint16_t* scales,
                  const uint8_t* zp, int n, int k, int group, const uint16_t* x, int m,
                  uint16_t* y, cudaStream_t s, bool pdl) {
  if (m == 1) {
    // three rows per warp when two would leave a second pass (and the
    // registers allow it): the whole layer is then requested before the wait
    if constexpr (CPL <= 4)
      if (n > 2 * kWarps * 2 * di.sms)
        return run<CPL, 1, 3>(di, codes, scales, zp, n, k, group, x, m, y, s, pdl);
    return run<CPL, 1, 2>(di, codes, scales, zp, n, k, group, x, m, y, s, pdl);
  }
  if (m == 2) return run<CPL, 2, 2>(di, codes, scales, zp, n, k, group, x, m, y, s, pdl);
  if (m <= 4) return run<CPL, 4, 2>(di, codes, scales, zp, n, k, group, x, m, y, s, pdl);
  return run<CPL, 8, 2>(di, codes, scales, zp, n, k, group, x, m, y, s, pdl);
}

}  // namespace

cudaError_t launch_int4_matvec(const uint8_t* codes, const uint16_t* scales, const uint8_t* zp,
                               int n, int k, int group, const uint16_t* x, int m, uint16_t* y,
                               cudaStream_t s, bool pdl) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorNoDevice;
  if (m == 1 && group == 128 && k <= 4096) {
    switch ((k + 1023) / 1024) {
      case 1: return run_mma_ppw<1>(*di, codes, scales, zp, n, k, x, y, s, pdl);
      case 2: return run_mma_ppw<2>(*di, codes, scales, zp, n, k, x, y, s, pdl);
      case 3: return run_mma_ppw<3>(*di, codes, scales, zp, n, k, x, y, s, pdl);
      default: return run_mma_ppw<4>(*di, codes, scales, zp, n, k, x, y, s, pdl);
    }
  }
  switch ((k / 32 + 31) / 32) {
    case 1: return run_m<1>(*di, codes, scales, zp, n, k, group, x, m, y, s, pdl);
    case 2: return run_m<2>(*di, codes, scales, zp, n, k, group, x, m, y, s, pdl);
    case 3: return run_m<3>(*di, codes, scales, zp, n, k, group, x, m, y, s, pdl);
    case 4: return run_m<4>(*di, codes, scales, zp, n, k, group, x, m, y, s, pdl);
    case 5: return run_m<5>(*di, codes, scales, zp, n, k, group, x, m, y, s, pdl);
    case 6: return run_m<6>(*di, codes, scales, zp, n, k, group, x, m, y, s, pdl);
    case 7: return run_m<7>(*di, codes, scales, zp, n, k, group, x, m, y, s, pdl);
    case 8: return run_m<8>(*di, codes, scales, zp, n, k, group, x, m, y, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tt
