// Router helpers and workspace layout shared by the MoE kernels: the
// compensated fp32 dot-product pieces, the warp top-k + softmax, and where
// the counters, router partials and SwiGLU outputs live in the workspace.
#pragma once

#include "common.cuh"

namespace tt {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kMaxRouterSplit = 8;  // router partial sums per expert (fused kernel)

// Workspace: [counters 64 B][router partials, one replica per CTA:
// kMaxMoeGrid x 256 x (s, c) fp32][output partials: kMaxMoeGrid x hidden
// fp32].  The whole workspace must be zero before the first call.  Counter 1
// (64-bit) advances by the grid size per call and is never reset; the router
// replicas mark an empty slot with zero bits and are cleared again by the
// CTA that reads them.
constexpr int kMaxMoeGrid = 256;
constexpr int kMaxRouterTasks = 256;  // E * split <= max(E, grid) <= 256
constexpr int kWsCounterBytes = 64;
constexpr int kWsRouterBytes = kMaxMoeGrid * kMaxRouterTasks * 8;
constexpr int kWsHOffset = kWsCounterBytes + kWsRouterBytes;

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

// One warp: the top_k largest logits (ties to the lower expert index), in
// descending order, and the softmax over them.  Logits must be finite.
__device__ __forceinline__ void warp_topk_softmax(const float* __restrict__ logits, int E, int top_k, int lane,
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


// The same for E <= 32 with one logit per lane (v: this lane's logit; lanes
// >= E are ignored).  Each lane counts the logits that beat its own (larger,
// or equal with a lower index) over 31 independent shuffles, which gives its
// rank in the total order; the ranks below top_k are the selection.  The
// softmax terms are summed in rank order, as in the general version.
__device__ __forceinline__ void warp_topk_softmax32(float v, int E, int top_k, int lane, int* idx,
                                                    float* prob) {
  const bool valid = lane < E;
  const float mv = valid ? v : -INFINITY;
  int rank = 0;
  float vmax = mv;
#pragma unroll
  for (int d = 1; d < 32; ++d) {
    const int o = (lane + d) & 31;
    const float ov = __shfl_sync(0xffffffffu, mv, o);
    const bool ovalid = o < E;
    rank += (ovalid && (ov > mv || (ov == mv && o < lane))) ? 1 : 0;
    vmax = fmaxf(vmax, ovalid ? ov : -INFINITY);
  }
  const bool sel = valid && rank < top_k;
  if (sel) idx[rank] = lane;
  const float ex = sel ? expf(mv - vmax) : 0.f;  // vmax: the rank-0 logit
  float den = 0.f;
  for (int j = 0; j < top_k; ++j) {
    const unsigned m = __ballot_sync(0xffffffffu, sel && rank == j);
    den += __shfl_sync(0xffffffffu, ex, __ffs(m) - 1);
  }
  if (sel) prob[rank] = ex / den;
}

}  // namespace tt
