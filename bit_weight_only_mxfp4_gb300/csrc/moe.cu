// MoE layer at batch 1: router -> top-k -> softmax over the selected experts
// -> only those experts' MXFP4 gate/up SwiGLU and down projections, summed
// with the router weights.
//
// Method: the ThinTensor pages route through router and expert stages
// (kerbin.cskartikey.dev/@satvikhardat, Dev Log #2 execution tape), run a
// block-scaled matvec over the *selected* experts only and insist on exact
// routing (stardance.hackclub.com/projects/29750: MoE drift devlog, "Hitting
// 100hrs and final ship"), with expert routing on the decode hot path.
//
// Three kernels chained with programmatic dependent launch:
//   moe_router_kernel   one CTA per expert: logit = x . W_r[e] summed with a
//                       compensated (two-float) fp32 sum, so the stored fp32
//                       logit is the rounding of the exact dot product; the
//                       top-k decision is taken on those fp32 values.
//   moe_gate_up_kernel  recomputes top-k + softmax (one warp), then streams the
//                       top_k * inter packed gate/up records of the selected
//                       experts (bulk copies into per-warp rings) and writes
//                       h_j = silu(g) * u in fp32 to the workspace.
//   moe_down_kernel     recomputes top-k from the logits (already complete when
//                       it starts), prefetches its down rows before waiting on
//                       the gate/up kernel, then out[r] = sum_j p_j * W_dn[e_j][r] . h_j
//                       with h_j split into an exact f16 hi + lo pair.
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "layout.cuh"
#include "mxfp4_core.cuh"

namespace tt {
namespace {

constexpr int kRouterThreads = 256;
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kLogitsBytes = kMaxExperts * 4;  // workspace: logits first

// Error-free sum: s + e == a + b exactly (Knuth's TwoSum; no contraction
// since only additions are involved, written with _rn intrinsics anyway).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// (s, c) += p with the rounding error of s carried in c.
__device__ __forceinline__ void comp_add(float& s, float& c, float p) {
  float t, e;
  two_sum(s, p, t, e);
  s = t;
  c = __fadd_rn(c, e);
}

__device__ __forceinline__ void comp_merge(float& s, float& c, float s2, float c2) {
  float t, e;
  two_sum(s, s2, t, e);
  s = t;
  c = __fadd_rn(__fadd_rn(c, c2), e);
}

__global__ void __launch_bounds__(kRouterThreads)
    moe_router_kernel(const uint16_t* __restrict__ x, int hidden, const uint16_t* __restrict__ wr,
                      float* __restrict__ logits) {
  __shared__ float red_s[kRouterThreads / 32], red_c[kRouterThreads / 32];
  pdl_allow_next_grid();   // the next kernel waits for this grid before reading logits
  pdl_wait_prior_grid();   // x is produced by the previous kernel
  const int e = blockIdx.x;
  const uint4* wv4 = reinterpret_cast<const uint4*>(wr + (size_t)e * hidden);
  const uint4* xv4 = reinterpret_cast<const uint4*>(x);
  float s = 0.f, c = 0.f;
  for (int t = threadIdx.x; t < (hidden >> 3); t += kRouterThreads) {
    const uint4 a = xv4[t];
    const uint4 b = __ldcs(wv4 + t);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      // bf16 x bf16 has at most 16 significant bits: exact in fp32
      comp_add(s, c, __fmul_rn(bf16_bits_to_f32(aw[q] & 0xFFFFu), bf16_bits_to_f32(bw[q] & 0xFFFFu)));
      comp_add(s, c, __fmul_rn(bf16_bits_to_f32(aw[q] >> 16), bf16_bits_to_f32(bw[q] >> 16)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
    comp_merge(s, c, s2, c2);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    red_s[warp] = s;
    red_c[warp] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float ts = red_s[0], tc = red_c[0];
    for (int w = 1; w < kRouterThreads / 32; ++w) comp_merge(ts, tc, red_s[w], red_c[w]);
    logits[e] = __fadd_rn(ts, tc);
  }
}

// One warp: the top_k largest logits (ties to the lower expert index), in
// descending order, and the softmax over them.  Logits must be finite.
__device__ void warp_topk_softmax(const float* __restrict__ logits, int E, int top_k, int lane,
                                  int* idx, float* prob) {
  float v[kMaxExperts / 32];
  bool taken[kMaxExperts / 32];
#pragma unroll
  for (int i = 0; i < kMaxExperts / 32; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? logits[e] : 0.f;
    taken[i] = e >= E;
  }
  float sel[kMaxTopK];
  for (int j = 0; j < top_k; ++j) {
    float bv = 0.f;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      const int e = lane + 32 * i;
      if (!taken[i] && (be == 0x7FFFFFFF || v[i] > bv)) {  // e increases with i
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      const bool take = oe != 0x7FFFFFFF && (be == 0x7FFFFFFF || ov > bv || (ov == bv && oe < be));
      if (take) {
        bv = ov;
        be = oe;
      }
    }
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i)
      if (lane + 32 * i == be) taken[i] = true;
    sel[j] = bv;
    if (lane == 0) idx[j] = be;
  }
  if (lane == 0) {
    float den = 0.f;
    float ex[kMaxTopK];
    for (int j = 0; j < top_k; ++j) {
      ex[j] = expf(sel[j] - sel[0]);  // sel[0] is the largest
      den += ex[j];
    }
    for (int j = 0; j < top_k; ++j) prob[j] = ex[j] / den;
  }
}

// ---------------------------------------------------------------------------
// Gathered gate/up SwiGLU over the selected experts.  Record q of the launch
// is row r = q % inter of selected expert j = q / inter; experts are stacked
// in `gate_up` at a stride of inter * SwigluRecord(hidden).bytes.  h_j[r] =
// silu(g) * u is written in fp32 (the experts carry no postscale: 1.0).
// ---------------------------------------------------------------------------
constexpr int kGuWarps = 16;
constexpr int kGuSlots = 2;

template <int NB>
__global__ void __launch_bounds__(kGuWarps * 32, 1)
    moe_gate_up_kernel(const uint16_t* __restrict__ x, int hidden, int inter, int E, int top_k,
                       const uint8_t* __restrict__ gate_up, const float* __restrict__ logits,
                       float* __restrict__ h_ws, int32_t* __restrict__ out_idx,
                       float* __restrict__ out_prob, int32_t* err) {
  constexpr int THREADS = kGuWarps * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const SwigluRecord L(hidden);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int total = top_k * inter;
  const int q0 = int((int64_t)total * blockIdx.x / gridDim.x);
  const int q1 = int((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  const int nitems = (q1 - q0) > warp ? (q1 - q0 - warp + kGuWarps - 1) / kGuWarps : 0;
  const size_t ring_bytes = (size_t)kGuWarps * kGuSlots * L.bytes;
  const int64_t expert_stride = (int64_t)inter * L.bytes;

  WarpRing ring;
  ring.slots = kGuSlots;
  ring.rec_bytes = L.bytes;
  ring.slot_bytes = L.bytes;
  ring.base = smem + (size_t)warp * kGuSlots * L.bytes;
  ring.bars = reinterpret_cast<uint64_t*>(smem + ring_bytes) + warp * kGuSlots;
  ring.packed = gate_up;  // record addresses are computed per expert below
  ring.policy = l2_evict_first_policy();
  uint4* xraw = reinterpret_cast<uint4*>(smem + ring_bytes + (size_t)kGuWarps * kGuSlots * 8);
  uint4* xs = xraw + (hidden >> 3);
  float* red = reinterpret_cast<float*>(xs + (hidden >> 3));
  int* sidx = reinterpret_cast<int*>(red + kGuWarps);
  float* sprob = reinterpret_cast<float*>(sidx + kMaxTopK);
  ring.init(lane);

  pdl_wait_prior_grid();  // logits (router) and x
  pdl_allow_next_grid();  // the down kernel may start: the router is complete
  if (warp == 0) warp_topk_softmax(logits, E, top_k, lane, sidx, sprob);
  __syncthreads();
  if (blockIdx.x == 0 && threadIdx.x < top_k) {
    out_idx[threadIdx.x] = sidx[threadIdx.x];
    out_prob[threadIdx.x] = sprob[threadIdx.x];
  }

  // record q -> its packed address (expert sidx[q / inter], row q % inter)
  auto rec_ptr = [&](int q) -> const uint8_t* {
    const int j = q / inter, r = q - j * inter;
    return gate_up + (int64_t)sidx[j] * expert_stride + (int64_t)r * L.bytes;
  };
  auto issue = [&](int t) {  // lane 0: item t of this warp -> slot t % slots
    const int q = q0 + warp + t * kGuWarps;
    const int s = t % kGuSlots;
    const uint32_t bar = smem_u32(&ring.bars[s]);
    mbar_arrive_expect_tx(bar, uint32_t(L.bytes));
    bulk_g2s(smem_u32(ring.base + (size_t)s * L.bytes), rec_ptr(q), uint32_t(L.bytes), bar,
             ring.policy);
  };
  if (lane == 0)
    for (int t = 0; t < min(kGuSlots, nitems); ++t) issue(t);

  // x -> f16 chunk-major in shared memory, one power-of-two prescale
  const int nchunk16 = hidden >> 3;
  float mx = 0.f;
  for (int c = threadIdx.x; c < nchunk16; c += THREADS) {
    const uint4 v = reinterpret_cast<const uint4*>(x)[c];
    xraw[c] = v;
    const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      mx = fmaxf(mx, fmaxf(fabsf(bf16_bits_to_f32(vw[e] & 0xFFFFu)),
                           fabsf(bf16_bits_to_f32(vw[e] >> 16))));
  }
  mx = warp_max(mx);
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  float gmax = red[0];
#pragma unroll
  for (int w = 1; w < kGuWarps; ++w) gmax = fmaxf(gmax, red[w]);
  const int sx = min(f16_prescale_exponent(gmax), 127);
  const float two_s = scalbnf(1.0f, sx);
  const float inv = scalbnf(1.0f, -sx);
  for (int c = threadIdx.x; c < nchunk16; c += THREADS) {
    const uint4 v = xraw[c];
    uint4 o;
    o.x = pack_f16x2_scaled(bf16_bits_to_f32(v.x & 0xFFFFu), bf16_bits_to_f32(v.x >> 16), two_s);
    o.y = pack_f16x2_scaled(bf16_bits_to_f32(v.y & 0xFFFFu), bf16_bits_to_f32(v.y >> 16), two_s);
    o.z = pack_f16x2_scaled(bf16_bits_to_f32(v.z & 0xFFFFu), bf16_bits_to_f32(v.z >> 16), two_s);
    o.w = pack_f16x2_scaled(bf16_bits_to_f32(v.w & 0xFFFFu), bf16_bits_to_f32(v.w >> 16), two_s);
    xs[(c & 3) * L.nblk + (c >> 2)] = o;
  }
  __syncthreads();

  float my_val = 0.f;
  int my_q = -1, fill = 0;
  for (int t = 0; t < nitems; ++t) {
    const uint8_t* rec = ring.wait(t);
    if (rec == nullptr) {
      if (lane == 0) flag_error(err, kErrTimeout);
      ring.drain(t, nitems);
      return;
    }
    float ag = 0.f, au = 0.f;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int b = 32 * i + lane;
      if (b < L.nblk) {
        uint32_t xv[16];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const uint4 tq = xs[qq * L.nblk + b];
          xv[4 * qq + 0] = tq.x;
          xv[4 * qq + 1] = tq.y;
          xv[4 * qq + 2] = tq.z;
          xv[4 * qq + 3] = tq.w;
        }
        const uint4 cg = *reinterpret_cast<const uint4*>(rec + L.gate_codes() + b * 16);
        const uint4 cu = *reinterpret_cast<const uint4*>(rec + L.up_codes() + b * 16);
        ag = fmaf(dot32(cg, xv), e8m0_to_f32(rec[L.gate_scales() + b]), ag);
        au = fmaf(dot32(cu, xv), e8m0_to_f32(rec[L.up_scales() + b]), au);
      }
    }
    const float pg = *reinterpret_cast<const float*>(rec + L.post);
    const float pu = *reinterpret_cast<const float*>(rec + L.post + 4);
    __syncwarp();
    if (lane == 0 && t + kGuSlots < nitems) issue(t + kGuSlots);
    const float v = warp_sum2(ag, au, lane);  // lanes 0-15: g, 16-31: u
    const float g = __shfl_sync(0xffffffffu, v, 0) * inv * pg;
    const float u = __shfl_sync(0xffffffffu, v, 16) * inv * pu;
    if (fill == 32) {  // batched epilogue: one record per lane
      if (my_q >= 0) h_ws[my_q] = my_val;
      fill = 0;
      my_q = -1;
    }
    if (lane == fill) {
      my_val = silu_mul(g, u);
      my_q = q0 + warp + t * kGuWarps;
    }
    ++fill;
  }
  if (my_q >= 0) h_ws[my_q] = my_val;
}

// ---------------------------------------------------------------------------
// Gathered down projection and weighted sum:
//   out[r] = sum_j p_j * (W_dn[e_j][r, :] . h_j)
// Experts' down matrices are stacked in `down` at a stride of
// hidden * RowRecord(inter).bytes.  One warp per output row; a ring slot
// holds the row's top_k records (one bulk copy each, one mbarrier).
// h_j (fp32) enters as hi + lo f16 after a per-expert power-of-two prescale:
// hi = f16(h * 2^s), lo = f16(h * 2^s - hi), which represents h to ~22 bits.
// ---------------------------------------------------------------------------
constexpr int kDnWarps = 8;
constexpr int kDnSlots = 2;

template <int NB>
__global__ void __launch_bounds__(kDnWarps * 32, 1)
    moe_down_kernel(int hidden, int inter, int E, int top_k, const uint8_t* __restrict__ down,
                    const float* __restrict__ logits, const float* __restrict__ h_ws,
                    uint16_t* __restrict__ out, int32_t* err) {
  constexpr int THREADS = kDnWarps * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const RowRecord L(inter);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r0 = int((int64_t)hidden * blockIdx.x / gridDim.x);
  const int r1 = int((int64_t)hidden * (blockIdx.x + 1) / gridDim.x);
  const int nitems = (r1 - r0) > warp ? (r1 - r0 - warp + kDnWarps - 1) / kDnWarps : 0;
  const int slot_bytes = top_k * L.bytes;
  const size_t ring_bytes = (size_t)kDnWarps * kDnSlots * slot_bytes;
  const int64_t expert_stride = (int64_t)hidden * L.bytes;
  const int nchunk16 = inter >> 3;

  uint8_t* base = smem + (size_t)warp * kDnSlots * slot_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ring_bytes) + warp * kDnSlots;
  uint4* xh = reinterpret_cast<uint4*>(smem + ring_bytes + (size_t)kDnWarps * kDnSlots * 8);
  // xh: [j][hi/lo][q][block] 16-byte chunks
  float* red = reinterpret_cast<float*>(xh + (size_t)top_k * 2 * nchunk16);  // [top_k][warps]
  float* scl = red + kMaxTopK * kDnWarps;                                    // [top_k] p_j * 2^-s_j
  int* sidx = reinterpret_cast<int*>(scl + kMaxTopK);
  float* sprob = reinterpret_cast<float*>(sidx + kMaxTopK);
  const uint64_t policy = l2_evict_first_policy();

  if (lane == 0) {
    for (int s = 0; s < kDnSlots; ++s) mbar_init(smem_u32(&bars[s]), 1);
    fence_mbar_init();
  }
  // The router grid completed before the gate/up kernel let this one launch,
  // so its logits can be read before waiting: pick the experts now and start
  // streaming their down rows while the gate/up kernel still runs.
  if (warp == 0) warp_topk_softmax(logits, E, top_k, lane, sidx, sprob);
  __syncthreads();
  auto issue = [&](int t) {  // lane 0: row r0 + warp + t*warps into slot t % slots
    const int r = r0 + warp + t * kDnWarps;
    const int s = t % kDnSlots;
    const uint32_t bar = smem_u32(&bars[s]);
    mbar_arrive_expect_tx(bar, uint32_t(slot_bytes));
    for (int j = 0; j < top_k; ++j)
      bulk_g2s(smem_u32(base + (size_t)s * slot_bytes + (size_t)j * L.bytes),
               down + (int64_t)sidx[j] * expert_stride + (int64_t)r * L.bytes, uint32_t(L.bytes),
               bar, policy);
  };
  if (lane == 0)
    for (int t = 0; t < min(kDnSlots, nitems); ++t) issue(t);
  pdl_allow_next_grid();
  pdl_wait_prior_grid();  // h from the gate/up kernel

  // h_j -> hi/lo f16 with a per-expert prescale (CTA-wide max per expert)
  for (int j = 0; j < top_k; ++j) {
    float mx = 0.f;
    for (int c = threadIdx.x; c < inter; c += THREADS) mx = fmaxf(mx, fabsf(h_ws[(size_t)j * inter + c]));
    mx = warp_max(mx);
    if (lane == 0) red[j * kDnWarps + warp] = mx;
  }
  __syncthreads();
  if (threadIdx.x < top_k) {
    float mx = 0.f;
    for (int w = 0; w < kDnWarps; ++w) mx = fmaxf(mx, red[threadIdx.x * kDnWarps + w]);
    const int sj = min(f16_prescale_exponent(mx), 127);
    red[threadIdx.x * kDnWarps] = __int_as_float(sj);  // stash the exponent
    scl[threadIdx.x] = sprob[threadIdx.x] * scalbnf(1.0f, -sj);
  }
  __syncthreads();
  for (int c = threadIdx.x; c < top_k * nchunk16; c += THREADS) {
    const int j = c / nchunk16, t8 = c - j * nchunk16;  // h_j[8*t8 .. 8*t8+7]
    const float two_s = scalbnf(1.0f, __float_as_int(red[j * kDnWarps]));
    const float4 a = reinterpret_cast<const float4*>(h_ws + (size_t)j * inter)[2 * t8];
    const float4 b = reinterpret_cast<const float4*>(h_ws + (size_t)j * inter)[2 * t8 + 1];
    const float v[8] = {a.x * two_s, a.y * two_s, a.z * two_s, a.w * two_s,
                        b.x * two_s, b.y * two_s, b.z * two_s, b.w * two_s};
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __half2 hh = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
      const float2 hf = __half22float2(hh);
      const __half2 ll = __floats2half2_rn(v[2 * e] - hf.x, v[2 * e + 1] - hf.y);
      hi[e] = *reinterpret_cast<const uint32_t*>(&hh);
      lo[e] = *reinterpret_cast<const uint32_t*>(&ll);
    }
    const int q = t8 & 3, blk = t8 >> 2;
    xh[(((size_t)j * 2 + 0) * 4 + q) * L.nblk + blk] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    xh[(((size_t)j * 2 + 1) * 4 + q) * L.nblk + blk] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
  __syncthreads();

  float my_val = 0.f;
  int my_r = -1, fill = 0;
  for (int t = 0; t < nitems; ++t) {
    const int s = t % kDnSlots;
    const bool ok = mbar_wait_bounded(smem_u32(&bars[s]), uint32_t((t / kDnSlots) & 1));
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) flag_error(err, kErrTimeout);
      const int issued = min(nitems, t + kDnSlots);
      for (int u = t + 1; u < issued; ++u)
        (void)mbar_wait_bounded(smem_u32(&bars[u % kDnSlots]), uint32_t((u / kDnSlots) & 1));
      return;
    }
    const uint8_t* slot = base + (size_t)s * slot_bytes;
    float acc = 0.f;
    for (int j = 0; j < top_k; ++j) {
      const uint8_t* rec = slot + (size_t)j * L.bytes;
      float aj = 0.f;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const int b = 32 * i + lane;
        if (b < L.nblk) {
          uint32_t hc[16], xv[16];
          decode32(*reinterpret_cast<const uint4*>(rec + L.codes() + b * 16), hc);
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const uint4 tq = xh[(((size_t)j * 2 + 0) * 4 + qq) * L.nblk + b];
            xv[4 * qq + 0] = tq.x;
            xv[4 * qq + 1] = tq.y;
            xv[4 * qq + 2] = tq.z;
            xv[4 * qq + 3] = tq.w;
          }
          float d = dot32_decoded(hc, xv);
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const uint4 tq = xh[(((size_t)j * 2 + 1) * 4 + qq) * L.nblk + b];
            xv[4 * qq + 0] = tq.x;
            xv[4 * qq + 1] = tq.y;
            xv[4 * qq + 2] = tq.z;
            xv[4 * qq + 3] = tq.w;
          }
          d += dot32_decoded(hc, xv);
          aj = fmaf(d, e8m0_to_f32(rec[L.scales() + b]), aj);
        }
      }
      acc = fmaf(aj, scl[j], acc);
    }
    __syncwarp();
    if (lane == 0 && t + kDnSlots < nitems) issue(t + kDnSlots);
    const float v = warp_sum(acc);
    if (fill == 32) {
      if (my_r >= 0) out[my_r] = f32_to_bf16_rne(my_val);
      fill = 0;
      my_r = -1;
    }
    if (lane == fill) {
      my_val = v;
      my_r = r0 + warp + t * kDnWarps;
    }
    ++fill;
  }
  if (my_r >= 0) out[my_r] = f32_to_bf16_rne(my_val);
}

template <typename Kern, typename... Args>
cudaError_t launch_ex(Kern kern, int grid, int threads, int smem, cudaStream_t s, bool pdl,
                      Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int NB>
cudaError_t run_gate_up(const DeviceInfo& di, const uint16_t* x, int hidden, int inter, int E,
                        int top_k, const uint8_t* gu, const float* logits, float* h_ws,
                        int32_t* out_idx, float* out_prob, cudaStream_t s, bool pdl) {
  const SwigluRecord L(hidden);
  const int smem = kGuWarps * kGuSlots * (L.bytes + 8) + 4 * hidden + kGuWarps * 4 +
                   kMaxTopK * 8 + 16;
  if (smem > di.smem_optin) return cudaErrorInvalidConfiguration;
  auto kern = moe_gate_up_kernel<NB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int total = top_k * inter;
  int grid = di.sms;
  const int need = (total + kGuWarps - 1) / kGuWarps;
  if (grid > need) grid = need;
  return launch_ex(kern, grid, kGuWarps * 32, smem, s, pdl, x, hidden, inter, E, top_k, gu,
                   logits, h_ws, out_idx, out_prob, di.error_word);
}

template <int NB>
cudaError_t run_down(const DeviceInfo& di, int hidden, int inter, int E, int top_k,
                     const uint8_t* dn, const float* logits, const float* h_ws, uint16_t* out,
                     cudaStream_t s, bool pdl) {
  const RowRecord L(inter);
  const int smem = kDnWarps * kDnSlots * (top_k * L.bytes + 8) + top_k * inter * 4 +
                   (kMaxTopK * kDnWarps + 3 * kMaxTopK) * 4 + 16;
  if (smem > di.smem_optin) return cudaErrorInvalidConfiguration;
  auto kern = moe_down_kernel<NB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int grid = di.sms;
  if (grid > hidden) grid = hidden;
  return launch_ex(kern, grid, kDnWarps * 32, smem, s, pdl, hidden, inter, E, top_k, dn, logits,
                   h_ws, out, di.error_word);
}

}  // namespace

size_t moe_workspace_bytes(int64_t hidden, int64_t inter, int n_experts, int top_k) {
  (void)hidden;
  (void)n_experts;
  return size_t(kLogitsBytes) + size_t(top_k) * size_t(inter) * 4;
}

cudaError_t launch_moe(const uint16_t* x, int hidden, int inter, const uint16_t* wr, int E,
                       int top_k, const uint8_t* gu, const uint8_t* dn, uint16_t* out,
                       int32_t* out_idx, float* out_prob, void* ws, cudaStream_t s, bool pdl) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorNoDevice;
  float* logits = static_cast<float*>(ws);
  float* h_ws = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kLogitsBytes);
  cudaError_t e = launch_ex(moe_router_kernel, E, kRouterThreads, 0, s, pdl, x, hidden, wr,
                            logits);
  if (e != cudaSuccess) return e;
  switch ((hidden / 32 + 31) / 32) {
#define TT_GU(nb) \
  case nb: e = run_gate_up<nb>(*di, x, hidden, inter, E, top_k, gu, logits, h_ws, out_idx, out_prob, s, true); break;
    TT_GU(1) TT_GU(2) TT_GU(3) TT_GU(4) TT_GU(5) TT_GU(6) TT_GU(7) TT_GU(8)
    TT_GU(9) TT_GU(10) TT_GU(11) TT_GU(12) TT_GU(13) TT_GU(14) TT_GU(15) TT_GU(16)
#undef TT_GU
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  switch ((inter / 32 + 31) / 32) {
#define TT_DN(nb) \
  case nb: e = run_down<nb>(*di, hidden, inter, E, top_k, dn, logits, h_ws, out, s, true); break;
    TT_DN(1) TT_DN(2) TT_DN(3) TT_DN(4) TT_DN(5) TT_DN(6) TT_DN(7) TT_DN(8)
#undef TT_DN
    default: return cudaErrorInvalidValue;
  }
  return e;
}

// ---------------------------------------------------------------------------
// Scratch for the MoE entry point that takes no workspace from its caller.
//
// Some callers cannot hand the library device memory: a plugin inside a host
// that owns the whole device pool and exposes no allocator, a real-time loop
// whose rules forbid allocator calls (they can synchronise the device or
// fragment the pool), or a binding with no access to a CUDA allocator.  For
// them the MoE layer runs on this fixed array instead: the router logits and
// the experts' fp32 SwiGLU outputs of one call: 1 KB + 32768 fp32 = 129 KB,
// enough for top_k * inter <= 32768 (gpt-oss-20b's 4 x 2880 uses 11520).
// Every GPU that loads the library holds it until the process exits.  All calls share it, so two such
// calls that overlap on the GPU (different streams, no ordering) race.
// Nothing in it needs clearing: each call writes every element it reads.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_moe_static_scratch[kLogitsBytes + kMoeStaticMaxHFloats * 4];

namespace {
std::mutex g_static_mu;
void* g_static_ptr[64];
}  // namespace

cudaError_t moe_static_scratch(void** ptr, size_t* bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    // Once per device, with that device current: the array's device address.
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_moe_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_ptr[dev] = p;
  }
  *ptr = g_static_ptr[dev];
  *bytes = sizeof(g_moe_static_scratch);
  return cudaSuccess;
}

}  // namespace tt
