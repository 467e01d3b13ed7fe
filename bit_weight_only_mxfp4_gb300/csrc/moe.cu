// MoE layer at batch 1: workspace sizing, the library-owned scratch of the
// workspace-free entry point, and dispatch to the single-kernel layer in
// moe_fused.cu.
//
// Method: the ThinTensor pages route through router and expert stages
// (kerbin.cskartikey.dev/@satvikhardat, Dev Log #2 execution tape), run a
// block-scaled matvec over the *selected* experts only and insist on exact
// routing (stardance.hackclub.com/projects/29750: MoE drift devlog, "Hitting
// 100hrs and final ship"), with expert routing on the decode hot path.
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "moe_common.cuh"

namespace tt {

size_t moe_workspace_bytes(int64_t hidden, int64_t inter, int n_experts, int top_k) {
  (void)inter;
  (void)n_experts;
  (void)top_k;
  return moe_fused_workspace_bytes(hidden);
}

cudaError_t launch_moe(const uint16_t* x, int hidden, int inter, const uint16_t* wr, int E,
                       int top_k, const uint8_t* const* gu, const uint8_t* const* dn,
                       uint16_t* out, int32_t* out_idx, float* out_prob, void* ws,
                       cudaStream_t s, bool pdl) {
  return launch_moe_fused(x, hidden, inter, wr, E, top_k, gu, dn, out, out_idx, out_prob, ws, s,
                          pdl);
}

// ---------------------------------------------------------------------------
// Scratch for the MoE entry point that takes no workspace from its caller.
//
// Some callers cannot hand the library device memory: a plugin inside a host
// that owns the whole device pool and exposes no allocator, a real-time loop
// whose rules forbid allocator calls (they can synchronise the device or
// fragment the pool), or a binding with no access to a CUDA allocator.  For
// them the MoE layer runs on this fixed array instead: the grid-wide
// counters, router partials and the per-CTA output partial sums of one call:
// 524,352 B + 256 x 4096 fp32 = 4.7 MB, enough for hidden <= 4096 (gpt-oss-20b
// uses 2880).  Static device memory starts zeroed, which is what the counters
// need.
// Every GPU that loads the library holds it until the process exits.  All calls share it, so two such
// calls that overlap on the GPU (different streams, no ordering) race.
// Each call writes every other element it reads, and leaves the counters at
// the next multiple of the grid size.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char
    g_moe_static_scratch[kWsHOffset + kMaxMoeGrid * kMoeStaticMaxHidden * 4];

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
