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
//                          once), a CTA per expert;
//   lowbit_swiglu_kernel   one CTA per (selected expert, 32 rows); every
//                          CTA takes the top-k + softmax from the logits,
//                          requests its rows' chunks (8 warps splitting k),
//                          builds the table of x meanwhile; h = silu(g) u
//                          in fp32 to the workspace;
//   lowbit_down_kernel     out = sum_j p_j down_j h_j: a cluster of top_k
//                          CTAs per 32 output rows, one per selected expert
//                          (its own table of h_j), the experts' rows summed
//                          in order through distributed shared memory.
#include <cmath>

#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "moe_common.cuh"
#include "mxfp4_core.cuh"

namespace tt {
namespace {

namespace cg = cooperative_groups;

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
// Router: a CTA per expert, its 8 warps splitting k in 8-element chunks (at
// most 4 per lane); products of bf16 are exact in fp32 and are summed with
// their rounding errors carried (TwoSum), the warps' sums merged in order,
// then rounded once.  The expert's weight row is requested before the wait.
// ---------------------------------------------------------------------------
constexpr int kRouterChunks = 4;  // 8-element chunks per lane (hidden <= 8192)

__global__ void __launch_bounds__(kLbThreads)
    lowbit_router_kernel(const uint16_t* __restrict__ x, int hidden,
                         const uint16_t* __restrict__ wr, int E, float* __restrict__ logits) {
  __shared__ float ps[kLbWarps], pc[kLbWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x;
  const int nch = hidden / 8, c0 = nch * warp / kLbWarps, c1 = nch * (warp + 1) / kLbWarps;
  const uint16_t* row = wr + int64_t(e) * hidden;
  uint4 a[kRouterChunks], b[kRouterChunks];
#pragma unroll
  for (int t = 0; t < kRouterChunks; ++t) {
    const int ch = c0 + lane + 32 * t;
    a[t] = ch < c1 ? __ldg(reinterpret_cast<const uint4*>(row) + ch) : make_uint4(0u, 0u, 0u, 0u);
  }
  pdl_allow_next_grid();
  pdl_wait_prior_grid();  // x comes from the preceding kernel
#pragma unroll
  for (int t = 0; t < kRouterChunks; ++t) {
    const int ch = c0 + lane + 32 * t;
    b[t] = ch < c1 ? __ldcg(reinterpret_cast<const uint4*>(x) + ch) : make_uint4(0u, 0u, 0u, 0u);
  }
  float s = 0.f, c = 0.f;
#pragma unroll
  for (int t = 0; t < kRouterChunks; ++t) {
    const uint32_t aw[4] = {a[t].x, a[t].y, a[t].z, a[t].w}, bw[4] = {b[t].x, b[t].y, b[t].z, b[t].w};
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
  if (lane == 0) {
    ps[warp] = s;
    pc[warp] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float ts = ps[0], tc = pc[0];
    for (int w2 = 1; w2 < kLbWarps; ++w2) comp_merge(ts, tc, ps[w2], pc[w2]);
    logits[e] = __fadd_rn(ts, tc);
  }
}

// Global -> shared copy of n float4 with up to U loads in flight per thread
// (NT threads).
template <int U, int NT>
__device__ __forceinline__ void stage_f4(float4* __restrict__ dst, const float4* __restrict__ src,
                                         int n, int tid) {
  for (int base = tid; base < n; base += U * NT) {
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * NT;
      if (i < n) v[u] = __ldcg(src + i);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * NT;
      if (i < n) dst[i] = v[u];
    }
  }
}

// The signed table of a vector v (length len, zero past it; len % 4 == 0):
// entry [g][nib] = ((s_0 v[4g] + s_1 v[4g+1]) + s_2 v[4g+2]) + s_3 v[4g+3],
// s_i = -1 where bit i of nib is set, for g over round_up(len, 128) / 4
// groups.  A thread per (group, top two sign bits): its 4 entries share
// s_2 and s_3; the 4 threads of a group read its values as one broadcast
// float4 and store consecutive 16-byte pieces (no bank conflicts).
__device__ __forceinline__ void build_sign_table(float* __restrict__ tab, int len,
                                                 const float* __restrict__ v, int tid,
                                                 int nthreads) {
  const int quads = (len + kLbBlock - 1) / kLbBlock * (kLbBlock / 4) * 4;
  for (int i = tid; i < quads; i += nthreads) {
    const int g = i >> 2, q = i & 3;
    const float4 a = 4 * g < len ? *reinterpret_cast<const float4*>(v + 4 * g)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
    const float sz = (q & 1) ? -a.z : a.z, sw = (q & 2) ? -a.w : a.w;
    float4 e;
    e.x = ((a.x + a.y) + sz) + sw;
    e.y = ((-a.x + a.y) + sz) + sw;
    e.z = ((a.x - a.y) + sz) + sw;
    e.w = ((-a.x - a.y) + sz) + sw;
    reinterpret_cast<float4*>(tab)[i] = e;
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

// A row's plane chunks and block scales for up to kLbMaxBlk consecutive
// blocks, requested in one go (the loads of a whole task are in flight
// before any of them is used).
constexpr int kLbMaxBlk = 4;

// Passes of kLbMaxBlk blocks that cover the largest per-warp block range
// (ceil(nb / 8) blocks): uniform over the CTA, since the passes hold
// barriers.
__device__ __forceinline__ int lb_passes(int nb, int warps) {
  const int most = (nb + warps - 1) / warps;
  const int p = (most + kLbMaxBlk - 1) / kLbMaxBlk;
  return p < 1 ? 1 : p;
}

template <int BITS>
struct RowChunks {
  uint4 c[BITS][kLbMaxBlk];
  uint32_t sc[kLbMaxBlk];
};

template <int BITS>
__device__ __forceinline__ void row_load(RowChunks<BITS>& rc, const uint8_t* __restrict__ buf,
                                         int64_t n, const LbLayout& L, int64_t r, int b0,
                                         int nblk) {
  const uint8_t* p0 = buf + r * L.P + 16 * b0;
  const uint8_t* sc = buf + BITS * n * L.P + r * L.S + b0;
#pragma unroll
  for (int i = 0; i < kLbMaxBlk; ++i) {
    if (i < nblk) {
#pragma unroll
      for (int p = 0; p < BITS; ++p)
        rc.c[p][i] = __ldg(reinterpret_cast<const uint4*>(p0 + p * n * L.P + 16 * i));
      rc.sc[i] = __ldg(sc + i);
    } else {
#pragma unroll
      for (int p = 0; p < BITS; ++p) rc.c[p][i] = make_uint4(0u, 0u, 0u, 0u);
      rc.sc[i] = 0u;
    }
  }
}

// The row's dot product over those blocks with the table (block b0 first).
template <int BITS>
__device__ __forceinline__ float row_compute(const RowChunks<BITS>& rc, int b0, int nblk,
                                             const float* __restrict__ tab) {
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kLbMaxBlk; ++i) {
    if (i < nblk) {
      const float* tb = tab + (b0 + i) * (16 * 32);
      float v;
      if (BITS == 1)
        v = chunk_sum(tb, rc.c[0][i]);
      else
        v = -(0.5f * chunk_sum(tb, rc.c[0][i]) + chunk_sum(tb, rc.c[BITS - 1][i]));
      acc = fmaf(v, e8m0_to_f32(rc.sc[i]), acc);
    }
  }
  return acc;
}

__device__ __forceinline__ bool usable(const uint8_t* p) {
  return p != nullptr && !(reinterpret_cast<uintptr_t>(p) & 15u);
}

// ---------------------------------------------------------------------------
// Selected-expert gate/up SwiGLU.  Tasks are (selected expert, 32 rows); a
// CTA takes tasks blockIdx.x, + gridDim.x, ...  After the routing it
// requests its first task's chunks, then stages x and builds the table while
// they arrive; each task's chunks are requested one task ahead (the first
// pass of k, all of it when hidden <= 32 * 128).  The warps' partial sums
// meet in a double-buffered shared array: one barrier per task.
// ---------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(kLbThreads, BITS == 1 ? 2 : 1)
    lowbit_swiglu_kernel(const uint16_t* __restrict__ x, int hidden, int inter,
                         const float* __restrict__ logits, int E, int top_k,
                         const uint8_t* const* __restrict__ gu_tab, int32_t* __restrict__ out_idx,
                         float* __restrict__ out_prob, float* __restrict__ h,
                         int32_t* __restrict__ err) {
  extern __shared__ __align__(16) float tab[];  // [groups][16], then x as fp32
  __shared__ int sidx[kMaxTopK];
  __shared__ float sprob[kMaxTopK];
  __shared__ float pg[2][kLbWarps][32], pu[2][kLbWarps][32];
  __shared__ const uint8_t* etab[kMaxExperts];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const LbLayout L(hidden);
  const int nb = int(L.nb);
  const int64_t rows = 2 * int64_t(inter);
  float* xs = tab + nb * 16 * 32;
  const int groups = inter / 32, tasks = top_k * groups;
  const int b0 = nb * warp / kLbWarps, b1 = nb * (warp + 1) / kLbWarps;
  const int passes = lb_passes(nb, kLbWarps);  // the same for every warp of the CTA
  auto pass_blocks = [&](int it) {
    const int p0 = b0 + kLbMaxBlk * it;
    return b1 - p0 < 0 ? 0 : (b1 - p0 < kLbMaxBlk ? b1 - p0 : kLbMaxBlk);
  };
  for (int e = tid; e < E; e += kLbThreads) etab[e] = gu_tab[e];  // weights: before the wait
  pdl_allow_next_grid();
  pdl_wait_prior_grid();  // the logits, and x
  if (warp == 0) {
    if (E <= 32)
      warp_topk_softmax32(lane < E ? __ldcg(logits + lane) : 0.f, E, top_k, lane, sidx, sprob);
    else
      warp_topk_softmax(logits, E, top_k, lane, sidx, sprob);
  }
  __syncthreads();
  if (blockIdx.x == 0 && tid < top_k) {
    out_idx[tid] = sidx[tid];
    out_prob[tid] = sprob[tid];
    const uint8_t* p = etab[sidx[tid]];
    if (!usable(p)) flag_error(err, p ? kErrAlign : kErrNull);
  }
  // a task's expert buffer (null when unusable) and row
  auto task_buf = [&](int task) {
    const uint8_t* p = etab[sidx[task / groups]];
    return usable(p) ? p : nullptr;
  };
  auto task_row = [&](int task) { return int64_t(task % groups) * 32 + lane; };
  RowChunks<BITS> cg, cu, ng, nu;
  int task = blockIdx.x;
  const uint8_t* buf = task < tasks ? task_buf(task) : nullptr;
  if (buf) {
    row_load<BITS>(cg, buf, rows, L, task_row(task), b0, pass_blocks(0));
    row_load<BITS>(cu, buf, rows, L, task_row(task) + inter, b0, pass_blocks(0));
  }
  // the table of x, built while the first chunks arrive
  for (int i0 = tid; i0 < hidden / 8; i0 += 4 * kLbThreads) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * kLbThreads;
      if (i < hidden / 8) v[u] = __ldcg(reinterpret_cast<const uint4*>(x) + i);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * kLbThreads;
      if (i < hidden / 8) {
        const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          xs[8 * i + 2 * q] = bf16_bits_to_f32(wv[q] & 0xFFFFu);
          xs[8 * i + 2 * q + 1] = bf16_bits_to_f32(wv[q] >> 16);
        }
      }
    }
  }
  __syncthreads();
  build_sign_table(tab, hidden, xs, tid, kLbThreads);
  __syncthreads();
  for (int t = 0; task < tasks; ++t, task += gridDim.x) {
    const int64_t r = task_row(task);
    const int next = task + gridDim.x;
    const uint8_t* nbuf = next < tasks ? task_buf(next) : nullptr;
    float g = 0.f, u = 0.f;
    for (int it = 0; it < passes; ++it) {
      const int nblk = pass_blocks(it);
      if (it > 0 && buf) {
        row_load<BITS>(cg, buf, rows, L, r, b0 + kLbMaxBlk * it, nblk);
        row_load<BITS>(cu, buf, rows, L, r + inter, b0 + kLbMaxBlk * it, nblk);
      }
      if (it == passes - 1 && nbuf) {  // the next task's first chunks
        row_load<BITS>(ng, nbuf, rows, L, task_row(next), b0, pass_blocks(0));
        row_load<BITS>(nu, nbuf, rows, L, task_row(next) + inter, b0, pass_blocks(0));
      }
      if (buf && nblk > 0) {
        g += row_compute<BITS>(cg, b0 + kLbMaxBlk * it, nblk, tab);
        u += row_compute<BITS>(cu, b0 + kLbMaxBlk * it, nblk, tab);
      }
    }
    pg[t & 1][warp][lane] = g;
    pu[t & 1][warp][lane] = u;
    __syncthreads();
    if (warp == 0) {
      float gs = pg[t & 1][0][lane], us = pu[t & 1][0][lane];
#pragma unroll
      for (int w2 = 1; w2 < kLbWarps; ++w2) {
        gs += pg[t & 1][w2][lane];
        us += pu[t & 1][w2][lane];
      }
      h[int64_t(task / groups) * inter + r] = silu_mul(gs, us);
    }
    cg = ng;
    cu = nu;
    buf = nbuf;
  }
}

// ---------------------------------------------------------------------------
// Weighted down projection of the selected experts: one thread-block
// cluster of top_k CTAs per 32 output rows; CTA rank j takes selected
// expert j: the table of h_j, p_j * (D_j h_j) for the 32 rows (8 warps
// splitting k; the first chunks requested before h_j is staged).  Rank 0
// sums the ranks' rows in rank order through distributed shared memory.
// ---------------------------------------------------------------------------
constexpr int kDnWarps = 8;
constexpr int kDnThreads = 32 * kDnWarps;

template <int BITS>
__global__ void __launch_bounds__(kDnThreads)
    lowbit_down_kernel(int hidden, int inter, int n_experts, int top_k,
                       const int32_t* __restrict__ idx, const float* __restrict__ prob,
                       const uint8_t* const* __restrict__ dn_tab, const float* __restrict__ h,
                       uint16_t* __restrict__ out, int32_t* __restrict__ err) {
  extern __shared__ __align__(16) float tab[];  // [groups][16], then h_j
  __shared__ float po[kDnWarps][32];
  __shared__ float part[32];  // this rank's rows, read by rank 0
  __shared__ const uint8_t* etab[kMaxExperts];
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = int(cluster.block_rank());  // the selected expert (cluster = top_k CTAs)
  const int64_t c = int64_t(blockIdx.x / top_k) * 32 + lane;  // output row
  const int64_t cr = c < hidden ? c : hidden - 1;             // rows past the end load a valid row
  const LbLayout L(inter);
  const int nb = int(L.nb);
  float* hs = tab + nb * 16 * 32;
  const int b0 = nb * warp / kDnWarps, b1 = nb * (warp + 1) / kDnWarps;
  const int passes = lb_passes(nb, kDnWarps);  // the same for every warp of the CTA
  auto pass_blocks = [&](int it) {
    const int p0 = b0 + kLbMaxBlk * it;
    return b1 - p0 < 0 ? 0 : (b1 - p0 < kLbMaxBlk ? b1 - p0 : kLbMaxBlk);
  };
  for (int e = tid; e < n_experts; e += kDnThreads) etab[e] = dn_tab[e];  // before the wait
  pdl_allow_next_grid();
  pdl_wait_prior_grid();  // h, the selection
  __syncthreads();
  const uint8_t* buf = etab[__ldcg(idx + j)];
  const float pj = __ldcg(prob + j);
  const bool ok = usable(buf);
  if (!ok && tid == 0 && blockIdx.x < top_k) flag_error(err, buf ? kErrAlign : kErrNull);
  RowChunks<BITS> cc;
  if (ok) row_load<BITS>(cc, buf, hidden, L, cr, b0, pass_blocks(0));
  stage_f4<8, kDnThreads>(reinterpret_cast<float4*>(hs),
                          reinterpret_cast<const float4*>(h + int64_t(j) * inter), inter / 4, tid);
  __syncthreads();
  build_sign_table(tab, inter, hs, tid, kDnThreads);
  __syncthreads();
  float acc = 0.f;
  for (int it = 0; it < passes; ++it) {
    const int nblk = pass_blocks(it);
    if (it > 0 && ok) row_load<BITS>(cc, buf, hidden, L, cr, b0 + kLbMaxBlk * it, nblk);
    if (ok && nblk > 0) acc += row_compute<BITS>(cc, b0 + kLbMaxBlk * it, nblk, tab);
  }
  po[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    float s2 = po[0][lane];
#pragma unroll
    for (int w2 = 1; w2 < kDnWarps; ++w2) s2 += po[w2][lane];
    part[lane] = pj * s2;
  }
  cluster.sync();  // every rank's rows are in place
  if (j == 0 && warp == 0) {
    float t = 0.f;
    for (int r = 0; r < top_k; ++r) t += cluster.map_shared_rank(part, r)[lane];
    if (c < hidden) out[c] = f32_to_bf16_rne(t);
  }
  cluster.sync();  // rank 0 has read every rank's rows
}

}  // namespace

size_t lowbit_matrix_bytes(int bits, int64_t n, int64_t k) { return size_t(LbLayout(k).bytes(bits, n)); }

int lowbit_table_smem_bytes(int64_t k) { return int(LbLayout(k).nb * 16 * 32 * 4 + k * 4); }

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
  const int smem_gu = lowbit_table_smem_bytes(hidden);
  const int smem_dn = lowbit_table_smem_bytes(inter);
  if (smem_gu > di->smem_optin || smem_dn > di->smem_optin) return cudaErrorInvalidConfiguration;
  int occ = 0;  // resident gate/up CTAs per SM
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
  // router: a CTA per expert
  cfg.gridDim = dim3(unsigned(E));
  cfg.dynamicSmemBytes = 0;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaError_t e = cudaLaunchKernelEx(&cfg, lowbit_router_kernel, x, hidden, wr, E, logits))
    return e;
  // gate/up SwiGLU of the selected experts, then the weighted down projection
  cfg.numAttrs = 1;
  if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kgu, kLbThreads, smem_gu))
    return e;
  const int tasks = top_k * (inter / 32);  // (selected expert, 32 rows)
  const int resident = (occ < 1 ? 1 : occ) * di->sms;
  cfg.gridDim = dim3(unsigned(tasks < resident ? tasks : resident));
  cfg.dynamicSmemBytes = smem_gu;
  if (cudaError_t e = cudaLaunchKernelEx(&cfg, kgu, x, hidden, inter,
                                         static_cast<const float*>(logits), E, top_k, gu, out_idx,
                                         out_prob, h, di->error_word))
    return e;
  // one cluster of top_k CTAs (one per selected expert) per 32 output rows
  cudaLaunchAttribute dattr[2];
  dattr[0] = attr[0];
  dattr[1].id = cudaLaunchAttributeClusterDimension;
  dattr[1].val.clusterDim.x = unsigned(top_k);
  dattr[1].val.clusterDim.y = 1;
  dattr[1].val.clusterDim.z = 1;
  cfg.attrs = dattr;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3(unsigned((hidden + 31) / 32 * top_k));
  cfg.blockDim = dim3(kDnThreads);
  cfg.dynamicSmemBytes = smem_dn;
  return cudaLaunchKernelEx(&cfg, kdn, hidden, inter, E, top_k,
                            static_cast<const int32_t*>(out_idx),
                            static_cast<const float*>(out_prob), dn, static_cast<const float*>(h),
                            out, di->error_word);
}

}  // namespace tt
