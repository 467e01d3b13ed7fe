// The MoE layer with Q1 / Q2 packed low-bit experts: quantiser, router,
// selected-expert gate/up SwiGLU and the weighted down projection.
//
// Method: ThinTensor project page (stardance.hackclub.com/projects/29750),
// the 97.87 tok/s notes (the MoE experts of layers 0:24 packed as 1-bit
// "Q1" structures, 9.52 GB of MXFP4 becoming 2.38 GB) and the final devlog
// (Q2 and Q1 quantizers; a low-bit selected-expert SwiGLU kernel).  The
// pages do not print the encoding; the one the 4x footprint fixes for an
// MX-style format is taken: one (Q1) or two (Q2) bits per weight and one
// E8M0 step 2^X per 128 weights along k (1 + 8/128 = 1.0625 bits against
// MXFP4's 4.25).  X is the power of two nearest the block's mean |w|; Q1
// stores the sign (value (1 - 2c) 2^X), Q2 q = clamp(floor(w / 2^X) + 2,
// 0, 3) (value (q - 1.5) 2^X).
//
// Matrix buffer [n][k]: plane 0 [n][P] (+ plane 1 [n][P] for Q2), then the
// scales [n][S]; P = 16 ceil(k/128) (bit kk % 8 of byte kk / 8 holds bit p
// of element kk's code), S = ceil(k/128) rounded up to 16.
//
// The dot products.  With s_i = 1 - 2 b_i (b_i a code bit), every 4
// consecutive activations give a 16-entry table E[nib] = sum_i s_i x_i
// (shared memory, built once per CTA from the vector).  A block of 128
// weights is then 32 table lookups per plane: Q1 contributes sum E[nib0],
// Q2 -(E[nib0] / 2 + E[nib1]) (q - 1.5 = -(s_0 / 2 + s_1)), times the
// block's exact 2^X.  A warp owns 32 rows (lane = row), so at every step
// its lanes read the same 16-entry row of the table: no bank conflicts.
//
// Kernels, chained by programmatic dependent launch:
//   lowbit_router_kernel   logits = Wr x (compensated fp32 sums, rounded
//                          once), a warp per expert;
//   lowbit_swiglu_kernel   every CTA takes the top-k + softmax from the
//                          logits; CTAs take (selected expert, 32 rows)
//                          tasks, their 8 warps splitting k; h = silu(g) u
//                          in fp32 to the workspace;
//   lowbit_down_kernel     out = sum_j p_j down_j h_j: per selected expert a
//                          table from h_j, 32 output rows per CTA, 8 warps
//                          splitting k, experts summed in order; bf16 out.
#include <cmath>

#include "common.cuh"
#include "launch.h"
#include "moe_common.cuh"
#include "mxfp4_core.cuh"

namespace tt {
namespace {

constexpr int kLbBlock = 128;
constexpr int kLbWarps = 8;
constexpr int kLbThreads = 32 * kLbWarps;
constexpr uint32_t kFullMask = 0xffffffffu;

struct LbLayout {
  int64_t nb, P, S;
  __host__ __device__ explicit LbLayout(int64_t k)
      : nb((k + kLbBlock - 1) / kLbBlock), P(16 * ((k + kLbBlock - 1) / kLbBlock)),
        S((((k + kLbBlock - 1) / kLbBlock) + 15) / 16 * 16) {}
  __host__ __device__ int64_t bytes(int bits, int64_t n) const { return n * (bits * P + S); }
};

// ---------------------------------------------------------------------------
// Quantiser: one thread per (row, block), the block's |w| summed in fp64 in
// k order (the same sum, hence the same step, as the definition's).
// ---------------------------------------------------------------------------
template <int BITS>
__global__ void quantize_lowbit_kernel(const float* __restrict__ w, int64_t n, int64_t k,
                                       uint8_t* __restrict__ buf, int32_t* __restrict__ status) {
  const LbLayout L(k);
  const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n * L.nb) return;
  const int64_t r = t / L.nb, b = t - r * L.nb;
  const float* src = w + r * k + b * kLbBlock;
  const int cnt = int(k - b * kLbBlock < kLbBlock ? k - b * kLbBlock : kLbBlock);
  double s = 0.0;
  bool bad = false;
  for (int i = 0; i < cnt; ++i) {
    const float v = src[i];
    if (!isfinite(v)) bad = true;
    s += fabs(double(v));
  }
  uint32_t planes[BITS][4];
#pragma unroll
  for (int p = 0; p < BITS; ++p) planes[p][0] = planes[p][1] = planes[p][2] = planes[p][3] = 0u;
  uint8_t* scale = buf + BITS * n * L.P + r * L.S + b;
  if (bad) {
    *scale = 0xFF;  // NaN step, zero codes
    if (status) atomicOr(status, kErrNonfinite);
  } else {
    int x = -127;
    if (s != 0.0) {
      const double m = s / double(cnt);
      int e;
      const double f = frexp(m, &e);  // m = f 2^e, f in [0.5, 1)
      x = (e - 1) + (2.0 * f > 1.5 ? 1 : 0);
      x = x < -127 ? -127 : (x > 127 ? 127 : x);
    }
    *scale = uint8_t(x + 127);
    const double inv = ldexp(1.0, -x);  // w / 2^x, exact
#pragma unroll
    for (int wq = 0; wq < 4; ++wq)
      for (int ii = 0; ii < 32 && 32 * wq + ii < cnt; ++ii) {
        const float v = src[32 * wq + ii];
        unsigned code;
        if (BITS == 1) {
          code = v < 0.0f ? 1u : 0u;
        } else {
          double q = floor(double(v) * inv) + 2.0;
          q = q < 0.0 ? 0.0 : (q > 3.0 ? 3.0 : q);
          code = unsigned(q);
        }
#pragma unroll
        for (int p = 0; p < BITS; ++p) planes[p][wq] |= ((code >> p) & 1u) << ii;
      }
  }
#pragma unroll
  for (int p = 0; p < BITS; ++p)
    *reinterpret_cast<uint4*>(buf + p * n * L.P + r * L.P + 16 * b) =
        make_uint4(planes[p][0], planes[p][1], planes[p][2], planes[p][3]);
  if (b == L.nb - 1)  // the scale row's padding
    for (int64_t i = L.nb; i < L.S; ++i) buf[BITS * n * L.P + r * L.S + i] = 0;
}

// ---------------------------------------------------------------------------
// Router: a warp per expert; products of bf16 are exact in fp32 and are
// summed with their rounding errors carried (TwoSum), then rounded once.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kLbThreads)
    lowbit_router_kernel(const uint16_t* __restrict__ x, int hidden,
                         const uint16_t* __restrict__ wr, int E, float* __restrict__ logits) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * kLbWarps + (threadIdx.x >> 5);
  pdl_allow_next_grid();
  pdl_wait_prior_grid();  // x comes from the preceding kernel
  if (e >= E) return;
  const uint16_t* row = wr + int64_t(e) * hidden;
  float s = 0.f, c = 0.f;
  for (int k0 = 8 * lane; k0 < hidden; k0 += 256) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(row + k0));
    const uint4 b = __ldcg(reinterpret_cast<const uint4*>(x + k0));
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      comp_add(s, c, __fmul_rn(bf16_bits_to_f32(aw[q] & 0xFFFFu), bf16_bits_to_f32(bw[q] & 0xFFFFu)));
      comp_add(s, c, __fmul_rn(bf16_bits_to_f32(aw[q] >> 16), bf16_bits_to_f32(bw[q] >> 16)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float s2 = __shfl_xor_sync(kFullMask, s, o), c2 = __shfl_xor_sync(kFullMask, c, o);
    comp_merge(s, c, s2, c2);
  }
  if (lane == 0) logits[e] = __fadd_rn(s, c);
}

// The signed table of a vector v (length len, zero past it): entry
// [g][nib] = sum_{i<4} (bit i of nib ? -v[4g+i] : v[4g+i]), for g over
// round_up(len, 128) / 4 groups.
__device__ __forceinline__ void build_sign_table(float* __restrict__ tab, int len,
                                                 const float* __restrict__ v, int tid,
                                                 int nthreads) {
  const int groups = (len + kLbBlock - 1) / kLbBlock * (kLbBlock / 4);
  for (int g = tid; g < groups; g += nthreads) {
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = 4 * g + i < len ? v[4 * g + i] : 0.f;
    float e[16];
    e[0] = ((a[0] + a[1]) + a[2]) + a[3];
#pragma unroll
    for (int nib = 1; nib < 16; ++nib) {
      const int low = (nib & 1) ? 0 : (nib & 2) ? 1 : (nib & 4) ? 2 : 3;  // lowest set bit
      e[nib] = e[nib & (nib - 1)] - 2.f * a[low];
    }
    float4* dst = reinterpret_cast<float4*>(tab + 16 * g);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_float4(e[4 * q], e[4 * q + 1], e[4 * q + 2], e[4 * q + 3]);
  }
}

// sum over one plane chunk (128 weights, 4 words) of table[g0 + i][nib_i].
__device__ __forceinline__ float chunk_sum(const float* __restrict__ tab, const uint4 c) {
  const uint32_t wv[4] = {c.x, c.y, c.z, c.w};
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      acc0 += tab[16 * (8 * q + i) + ((wv[q] >> (4 * i)) & 15u)];
      acc1 += tab[16 * (8 * q + i + 1) + ((wv[q] >> (4 * i + 4)) & 15u)];
    }
  }
  return acc0 + acc1;
}

// One row's dot product with a table over blocks [b0, b1) of a matrix
// buffer (row r of n, k's layout L).
template <int BITS>
__device__ __forceinline__ float row_dot(const uint8_t* __restrict__ buf, int64_t n,
                                         const LbLayout& L, int64_t r, int b0, int b1,
                                         const float* __restrict__ tab) {
  float acc = 0.f;
  const uint8_t* p0 = buf + r * L.P;
  const uint8_t* sc = buf + BITS * n * L.P + r * L.S;
  for (int b = b0; b < b1; ++b) {
    const float* tb = tab + b * (16 * 32);
    const float scale = e8m0_to_f32(__ldg(sc + b));
    const uint4 c0 = __ldg(reinterpret_cast<const uint4*>(p0 + 16 * b));
    float v;
    if (BITS == 1) {
      v = chunk_sum(tb, c0);
    } else {
      const uint4 c1 = __ldg(reinterpret_cast<const uint4*>(p0 + n * L.P + 16 * b));
      v = -(0.5f * chunk_sum(tb, c0) + chunk_sum(tb, c1));
    }
    acc = fmaf(v, scale, acc);
  }
  return acc;
}

// ---------------------------------------------------------------------------
// Selected-expert gate/up SwiGLU.
// ---------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(kLbThreads)
    lowbit_swiglu_kernel(const uint16_t* __restrict__ x, int hidden, int inter,
                         const float* __restrict__ logits, int E, int top_k,
                         const uint8_t* const* __restrict__ gu_tab, int32_t* __restrict__ out_idx,
                         float* __restrict__ out_prob, float* __restrict__ h,
                         int32_t* __restrict__ err) {
  extern __shared__ __align__(16) float tab[];  // [groups][16], then x as fp32
  __shared__ int sidx[kMaxTopK];
  __shared__ float sprob[kMaxTopK];
  __shared__ const uint8_t* sbuf[kMaxTopK];
  __shared__ float pg[kLbWarps][32], pu[kLbWarps][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const LbLayout L(hidden);
  const int nb = int(L.nb);
  const int64_t rows = 2 * int64_t(inter);
  float* xs = tab + nb * 16 * 32;
  pdl_allow_next_grid();
  pdl_wait_prior_grid();  // the logits, and x
  if (warp == 0) {
    if (E <= 32)
      warp_topk_softmax32(lane < E ? __ldcg(logits + lane) : 0.f, E, top_k, lane, sidx, sprob);
    else
      warp_topk_softmax(logits, E, top_k, lane, sidx, sprob);
  }
  for (int i = tid; i < hidden; i += kLbThreads) xs[i] = bf16_bits_to_f32(x[i]);
  __syncthreads();
  if (tid < top_k) {
    const uint8_t* p = gu_tab[sidx[tid]];
    sbuf[tid] = p;
    if (p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u)) flag_error(err, p ? kErrAlign : kErrNull);
    if (blockIdx.x == 0) {
      out_idx[tid] = sidx[tid];
      out_prob[tid] = sprob[tid];
    }
  }
  build_sign_table(tab, hidden, xs, tid, kLbThreads);
  __syncthreads();
  // each warp: a contiguous range of the blocks
  const int b0 = nb * warp / kLbWarps, b1 = nb * (warp + 1) / kLbWarps;
  const int groups = inter / 32, tasks = top_k * groups;
  for (int task = blockIdx.x; task < tasks; task += gridDim.x) {
    const int j = task / groups, r = (task - j * groups) * 32 + lane;
    const uint8_t* buf = sbuf[j];
    float g = 0.f, u = 0.f;
    if (buf != nullptr && !(reinterpret_cast<uintptr_t>(buf) & 15u)) {
      g = row_dot<BITS>(buf, rows, L, r, b0, b1, tab);
      u = row_dot<BITS>(buf, rows, L, r + inter, b0, b1, tab);
    }
    pg[warp][lane] = g;
    pu[warp][lane] = u;
    __syncthreads();
    if (warp == 0) {
      float gs = pg[0][lane], us = pu[0][lane];
#pragma unroll
      for (int w2 = 1; w2 < kLbWarps; ++w2) {
        gs += pg[w2][lane];
        us += pu[w2][lane];
      }
      h[int64_t(j) * inter + r] = silu_mul(gs, us);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Weighted down projection of the selected experts.
// ---------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(kLbThreads)
    lowbit_down_kernel(int hidden, int inter, int top_k, const int32_t* __restrict__ idx,
                       const float* __restrict__ prob, const uint8_t* const* __restrict__ dn_tab,
                       const float* __restrict__ h, uint16_t* __restrict__ out,
                       int32_t* __restrict__ err) {
  extern __shared__ __align__(16) float tab[];  // [groups][16], then h_j as fp32
  __shared__ float po[kLbWarps][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const LbLayout L(inter);
  const int nb = int(L.nb);
  float* hs = tab + nb * 16 * 32;
  const int b0 = nb * warp / kLbWarps, b1 = nb * (warp + 1) / kLbWarps;
  const int64_t c = int64_t(blockIdx.x) * 32 + lane;  // output row
  pdl_allow_next_grid();
  pdl_wait_prior_grid();  // h, the selection
  float acc = 0.f;
  for (int j = 0; j < top_k; ++j) {
    const int e = __ldcg(idx + j);
    const float pj = __ldcg(prob + j);
    const uint8_t* buf = dn_tab[e];
    const bool ok = buf != nullptr && !(reinterpret_cast<uintptr_t>(buf) & 15u);
    if (!ok && tid == 0 && blockIdx.x == 0) flag_error(err, buf ? kErrAlign : kErrNull);
    __syncthreads();  // the previous expert's table is no longer read
    for (int i = tid; i < inter; i += kLbThreads) hs[i] = __ldcg(h + int64_t(j) * inter + i);
    __syncthreads();
    build_sign_table(tab, inter, hs, tid, kLbThreads);
    __syncthreads();
    if (ok && c < hidden) acc = fmaf(pj, row_dot<BITS>(buf, hidden, L, c, b0, b1, tab), acc);
  }
  po[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && c < hidden) {
    float s = po[0][lane];
#pragma unroll
    for (int w2 = 1; w2 < kLbWarps; ++w2) s += po[w2][lane];
    out[c] = f32_to_bf16_rne(s);
  }
}

}  // namespace

size_t lowbit_matrix_bytes(int bits, int64_t n, int64_t k) { return size_t(LbLayout(k).bytes(bits, n)); }

int lowbit_table_smem_bytes(int64_t k) {
  const LbLayout L(k);
  return int(L.nb * 16 * 32 * 4 + ((k + 3) / 4) * 16);
}

cudaError_t launch_quantize_lowbit(int bits, const float* w, int64_t n, int64_t k, uint8_t* buf,
                                   int32_t* status, cudaStream_t s) {
  const int64_t tasks = n * LbLayout(k).nb;
  if (tasks == 0) return cudaSuccess;
  const int threads = 128;
  const unsigned grid = unsigned((tasks + threads - 1) / threads);
  if (bits == 1)
    quantize_lowbit_kernel<1><<<grid, threads, 0, s>>>(w, n, k, buf, status);
  else
    quantize_lowbit_kernel<2><<<grid, threads, 0, s>>>(w, n, k, buf, status);
  return cudaGetLastError();
}

cudaError_t launch_moe_lowbit(int bits, const uint16_t* x, int hidden, int inter,
                              const uint16_t* wr, int E, int top_k, const uint8_t* const* gu,
                              const uint8_t* const* dn, uint16_t* out, int32_t* out_idx,
                              float* out_prob, void* ws, cudaStream_t s, bool pdl) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorNoDevice;
  float* h = static_cast<float*>(ws);
  float* logits = h + int64_t(top_k) * inter;
  const int smem_gu = lowbit_table_smem_bytes(hidden), smem_dn = lowbit_table_smem_bytes(inter);
  if (smem_gu > di->smem_optin || smem_dn > di->smem_optin) return cudaErrorInvalidConfiguration;
  auto kgu = bits == 1 ? lowbit_swiglu_kernel<1> : lowbit_swiglu_kernel<2>;
  auto kdn = bits == 1 ? lowbit_down_kernel<1> : lowbit_down_kernel<2>;
  if (cudaError_t e = ensure_smem(*di, kgu, smem_gu)) return e;
  if (cudaError_t e = ensure_smem(*di, kdn, smem_dn)) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.stream = s;
  cfg.blockDim = dim3(kLbThreads);
  // router
  cfg.gridDim = dim3(unsigned((E + kLbWarps - 1) / kLbWarps));
  cfg.dynamicSmemBytes = 0;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaError_t e = cudaLaunchKernelEx(&cfg, lowbit_router_kernel, x, hidden, wr, E, logits))
    return e;
  // gate/up SwiGLU of the selected experts, then the weighted down projection
  cfg.numAttrs = 1;
  const int tasks = top_k * (inter / 32);
  cfg.gridDim = dim3(unsigned(tasks < di->sms ? tasks : di->sms));
  cfg.dynamicSmemBytes = smem_gu;
  if (cudaError_t e = cudaLaunchKernelEx(&cfg, kgu, x, hidden, inter,
                                         static_cast<const float*>(logits), E, top_k, gu, out_idx,
                                         out_prob, h, di->error_word))
    return e;
  cfg.gridDim = dim3(unsigned((hidden + 31) / 32));
  cfg.dynamicSmemBytes = smem_dn;
  return cudaLaunchKernelEx(&cfg, kdn, hidden, inter, top_k, static_cast<const int32_t*>(out_idx),
                            static_cast<const float*>(out_prob), dn, static_cast<const float*>(h),
                            out, di->error_word);
}

}  // namespace tt
