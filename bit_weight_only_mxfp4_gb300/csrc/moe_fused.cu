// MoE layer at batch 1 as ONE persistent kernel: router -> top-k -> softmax
// -> the selected experts' gate/up SwiGLU -> their down projections, summed
// with the router weights.
//
// Method: the ThinTensor pages route on the device (kerbin.cskartikey.dev/
// @satvikhardat, Dev Log #2 execution tape: router and expert stages), run
// the block-scaled matvec over the *selected* experts only and insist on
// exact routing (stardance.hackclub.com/projects/29750: MoE drift devlog,
// "Hitting 100hrs and final ship").
//
// A layer moves ~53 MB at gpt-oss-20b sizes, a few microseconds of HBM time,
// so the dependent steps must not each pay a launch, a ramp-up and a drain,
// and no SM may wait for data that another SM produces if it can be avoided.
// One cooperative grid of one CTA per SM:
//
//   A  router: CTA c computes compensated partial dot products x . W_r[e]
//      over a slice of hidden (E * split tasks) and writes them into every
//      CTA's replica, where a written value marks itself (never all-zero
//      bits); every CTA polls its replica, folds each expert's partials in a
//      fixed order into the fp32 logit and takes the top-k + softmax itself.
//   B  the selected experts' SwiGLU outputs h (top_k * inter values) are
//      split into 16-wide slices; CTA c owns slices [hb0, hb1) and streams
//      exactly the gate/up records that produce them (per-warp bulk-copy
//      rings), keeping its h in shared memory.  At the same moment it
//      requests the matching COLUMN slices of the down matrices (packed by
//      column slice, so each is one contiguous run) for all hidden rows.
//   C  every warp streams its gate/up records free-running; after each
//      record it checks (without blocking) whether the next 16-wide slice of
//      h is complete and its down columns have landed, and if so multiplies
//      that slice into the down columns for the output rows it owns (rows
//      fixed per thread, so the sums are deterministic; h in fp32, packed
//      f32x2 FMAs, p_j folded in).  The down work thus fills the gaps of the
//      streaming, and only the last slice is left after it.  No h leaves the
//      SM that computed it; each CTA ends with one fp32 partial vector over
//      the hidden rows.
//   D  after grid counter 1, CTA c gathers the partial vectors of its output
//      rows into shared memory, sums them in a fixed order and rounds them
//      to bf16.
//
// Every wait (counters, mbarriers) is bounded in time; a timeout sets the
// library's error word and the CTA leaves after its own copies have landed.
#include <atomic>

#include "common.cuh"
#include "launch.h"
#include "layout.cuh"
#include "moe_common.cuh"
#include "mxfp4_core.cuh"

namespace tt {
namespace {

constexpr int kFWarps = 16;
constexpr int kFThreads = kFWarps * 32;
constexpr int kMaxGuSlots = 2;
constexpr int kMaxXChunksPerThread = 2;  // hidden <= 8192: 1024 chunks / 512 threads
constexpr int kRowsPerThread = 8;        // output rows per thread and row chunk
constexpr int kMaxChunkRows = kFThreads * kRowsPerThread;  // 4096
constexpr int kMaxDSlots = 32;           // down-item slots
constexpr int kMaxSlices = 32;           // 16-wide h slices per CTA

// Host-chosen launch plan; the same numbers fix the shared-memory carve-up.
struct MoePlan {
  int G;        // CTAs (one per SM)
  int nhb_max;  // max 16-wide h slices per CTA
  int gslots;   // gate/up ring slots per warp
  int rc;       // output rows per down item: hidden, or a multiple of 512
  int nchunk;   // ceil(hidden / rc)
  int item;     // bytes of a down item slot: rc * 8 codes + rc scales
  int dslots;   // down item slots
  // shared-memory offsets
  int bars, misc, tab, hs, xs, dring, gring, total;
};

__host__ __device__ inline int align128(int o) { return (o + 127) & ~127; }

__host__ __device__ inline void plan_offsets(MoePlan& p, int hidden, int gu_rec_bytes) {
  int o = 0;
  p.bars = o;  // gate/up ring, down slots, h slices
  o += (kFWarps * kMaxGuSlots + kMaxDSlots + kMaxSlices) * 8;
  p.misc = o;  // reductions, top-k, flags, per-slot consumer counts
  o += (2 * kFWarps + 2 * kMaxTopK + kMaxExperts + 4 + kMaxDSlots) * 4;
  o = (o + 7) & ~7;
  p.tab = o;  // the experts' gate/up and down pointers
  o += 2 * kMaxExperts * 8;
  p.hs = o;
  o += p.nhb_max * 16 * 4;
  o = align128(o);
  p.xs = o;
  o += hidden * 2;
  o = align128(o);
  p.dring = o;
  o += p.dslots * p.item;
  o = align128(o);
  p.gring = o;
  o += kFWarps * p.gslots * gu_rec_bytes;
  p.total = o;
}

// Largest plan that fits: as many gate/up slots per warp as possible (up to
// 2), down items as large as possible (whole columns when hidden <= 4096)
// with two slots or more, and as many slots as there are items if they fit.
// The phase-D gather reuses the rings and must fit in them.
bool make_plan(int hidden, int inter, int top_k, int G, int smem_limit, MoePlan& p) {
  const SwigluRecord Lg(hidden);
  const int HB = top_k * inter / 16;
  p.G = G;
  p.nhb_max = (HB + G - 1) / G;
  if (p.nhb_max > kMaxSlices) return false;
  const int rows_out = (hidden + G - 1) / G;
  for (int gs = kMaxGuSlots; gs >= 1; --gs) {
    int rc = hidden <= kMaxChunkRows ? hidden : kMaxChunkRows;
    while (rc >= kFThreads || rc == hidden) {
      p.gslots = gs;
      p.rc = rc;
      p.nchunk = (hidden + rc - 1) / rc;
      p.item = rc * 9;
      const int nitems = p.nchunk * p.nhb_max;
      p.dslots = 0;
      plan_offsets(p, hidden, Lg.bytes);
      const int room = smem_limit - p.total;
      int ds = room > 0 ? room / p.item : 0;
      if (ds > nitems) ds = nitems;
      if (ds > kMaxDSlots) ds = kMaxDSlots;
      if (ds >= 2 || (ds == 1 && nitems == 1)) {
        p.dslots = ds;
        plan_offsets(p, hidden, Lg.bytes);
        if (p.total - p.dring >= G * rows_out * 4 && p.total <= smem_limit) return true;
      }
      // next smaller item: a multiple of 512 rows, so each thread's rows
      // (t + 512 m) fall in whole chunks
      const int next = ((rc - 1) / kFThreads) * kFThreads;
      if (next < kFThreads) break;
      rc = next;
    }
  }
  return false;
}

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// *p += v with release semantics at GPU scope: the writes this CTA made
// before the preceding __syncthreads are visible to whoever acquires *p.
__device__ __forceinline__ void red_release_add(uint64_t* p, uint64_t v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Spins (bounded in time) until *p >= target.  One thread per CTA (the
// others wait at a barrier, so the poll takes no issue slots from work and
// does not sleep between loads); the acquire load orders the reads that
// follow it (with the __syncthreads that comes after, for the whole CTA).
__device__ bool wait_counter(const uint64_t* p, uint64_t target) {
  if (ld_acquire_u64(p) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ld_acquire_u64(p) >= target) return true;
    if ((it & 63u) == 0u && globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Router partials carry their own "written" mark: a stored value never has
// all-zero bits (+0.0 is stored as -0.0, which is equal in every sum), so a
// zero word is an empty slot.  The workspace starts zeroed, and each CTA
// clears its replica after reading it, for the next call.
__device__ __forceinline__ float nonzero_bits(float v) {
  return __float_as_uint(v) == 0u ? -0.0f : v;
}
__device__ __forceinline__ float2 ld_relaxed_f2(const float2* p) {
  float2 v;
  asm volatile("ld.relaxed.gpu.global.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_f2(float2* p, float2 v) {
  asm volatile("st.relaxed.gpu.global.v2.f32 [%0], {%1, %2};" ::"l"(p), "f"(v.x), "f"(v.y)
               : "memory");
}
// Polls `n` partials until every one has been written (bounded in time);
// one warp polls while the rest of the CTA waits at a barrier.
__device__ bool poll_partials(const float2* p, int n, float2* v) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    bool all = true;
#pragma unroll
    for (int q = 0; q < kMaxRouterSplit; ++q)
      if (q < n) {
        v[q] = ld_relaxed_f2(p + q);
        all = all && __float_as_uint(v[q].x) != 0u && __float_as_uint(v[q].y) != 0u;
      }
    if (all) return true;
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Bounded mbarrier wait that suspends the thread (up to hint_ns per try)
// instead of spinning, so waiting warps leave the issue slots to the warps
// that compute.
__device__ __forceinline__ bool mbar_wait_sleep_bounded(uint32_t bar, uint32_t parity,
                                                        uint32_t hint_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_sleep(bar, parity, hint_ns)) return true;
    if ((it & 15u) == 0u && globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// a += w * x on two fp32 lanes (one packed FMA; each lane an IEEE fma).
__device__ __forceinline__ void ffma2(float& a0, float& a1, float w0, float w1, float x0,
                                      float x1) {
  asm("{\n\t.reg .b64 A, W, X;\n\t"
      "mov.b64 A, {%0, %1};\n\t"
      "mov.b64 W, {%2, %3};\n\t"
      "mov.b64 X, {%4, %5};\n\t"
      "fma.rn.f32x2 A, W, X, A;\n\t"
      "mov.b64 {%0, %1}, A;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(w0), "f"(w1), "f"(x0), "f"(x1));
}

// 16 E2M1 codes (8 bytes, even k in the low nibble) dotted with 16 fp32
// values: codes widened exactly to f16 then f32, fp32 accumulation.
__device__ __forceinline__ float dot16_f32(const uint2& c, const float* hv) {
  uint32_t h[8];
  e2m1x8_to_f16x2(c.x, h[0], h[1], h[2], h[3]);
  e2m1x8_to_f16x2(c.y, h[4], h[5], h[6], h[7]);
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
    const float2 q = __half22float2(*reinterpret_cast<const __half2*>(&h[i + 1]));
    ffma2(a0, a1, p.x, p.y, hv[2 * i], hv[2 * i + 1]);
    ffma2(a2, a3, q.x, q.y, hv[2 * i + 2], hv[2 * i + 3]);
  }
  return (a0 + a1) + (a2 + a3);
}

// KH, KI: hidden and inter when fixed at compile time (0: the runtime
// arguments), which turns the record, slice and x offsets into immediates.
template <int NBG, int KH, int KI>
__global__ void __launch_bounds__(kFThreads, 1)
    moe_fused_kernel(const uint16_t* __restrict__ x, int hidden_arg, int inter_arg,
                     const uint16_t* __restrict__ wr, int E, int top_k,
                     const uint8_t* const* __restrict__ gu_tab,
                     const uint8_t* const* __restrict__ dn_tab, uint16_t* __restrict__ out,
                     int32_t* __restrict__ out_idx,
                     float* __restrict__ out_prob, uint8_t* __restrict__ ws, int split,
                     MoePlan P, int32_t* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int hidden = KH > 0 ? KH : hidden_arg;
  const int inter = KI > 0 ? KI : inter_arg;
  // With hidden fixed, the host launches this instance only with whole-
  // column down items (P.rc == hidden, one row chunk): the rows each thread
  // owns, and which of them exist, are then known at compile time.
  constexpr bool kOneChunk = KH > 0 && KH <= kMaxChunkRows;
  const int rc = kOneChunk ? KH : P.rc;
  const SwigluRecord Lg(hidden);
  const ColSlices Ld(hidden, inter);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G = gridDim.x;
  const int c = blockIdx.x;

  uint64_t* cnt = reinterpret_cast<uint64_t*>(ws);  // [1]: partial vectors ([0] unused)
  float2* part = reinterpret_cast<float2*>(ws + kWsCounterBytes);  // [G][T] replicas
  float* opart = reinterpret_cast<float*>(ws + kWsHOffset);        // [G][hidden]

  uint64_t* gbars = reinterpret_cast<uint64_t*>(smem + P.bars);  // [kFWarps][kMaxGuSlots]
  uint64_t* dbars = gbars + kFWarps * kMaxGuSlots;               // [kMaxDSlots]
  uint64_t* hbars = dbars + kMaxDSlots;                          // [kMaxSlices]: h slice ready
  float* red_s = reinterpret_cast<float*>(smem + P.misc);
  float* red_c = red_s + kFWarps;
  int* sidx = reinterpret_cast<int*>(red_c + kFWarps);
  float* sprob = reinterpret_cast<float*>(sidx + kMaxTopK);
  float* slog = sprob + kMaxTopK;
  int* sflag = reinterpret_cast<int*>(slog + kMaxExperts);
  int* sfail = sflag + 1;
  int* d_issued = sflag + 2;                        // down items issued so far
  int* dcons = sflag + 4;                           // [kMaxDSlots] warps done with the slot
  float* hs = reinterpret_cast<float*>(smem + P.hs);
  uint4* xs = reinterpret_cast<uint4*>(smem + P.xs);
  uint8_t* dring = smem + P.dring;
  uint8_t* gring = smem + P.gring;
  const uint8_t** tab_g = reinterpret_cast<const uint8_t**>(smem + P.tab);  // [E]
  const uint8_t** tab_d = tab_g + kMaxExperts;                             // [E]

  const int nch = hidden >> 3;
  const int HB = top_k * inter / 16;
  const int spe = inter >> 4;  // h slices per expert
  auto hb_lo = [&](int cc) { return int((int64_t)HB * cc / G); };
  const int hb0 = hb_lo(c), hb1 = hb_lo(c + 1);
  const int nhb = hb1 - hb0;  // rounds: every warp computes one record per round
  const int qa = hb0 * 16;
  const int T = E * split;
  const int cs = (nch + split - 1) / split;
  const uint64_t policy = l2_evict_first_policy();

  if (lane == 0) {
    for (int s = 0; s < P.gslots; ++s) mbar_init(smem_u32(&gbars[warp * kMaxGuSlots + s]), 1);
    for (int s = warp; s < P.dslots; s += kFWarps) {
      mbar_init(smem_u32(&dbars[s]), 1);
      dcons[s] = 0;
    }
    for (int s = warp; s < nhb; s += kFWarps) mbar_init(smem_u32(&hbars[s]), 16);  // 16 records
    if (warp == 0) {
      *sfail = 0;
      *d_issued = 0;
    }
    fence_mbar_init();
  }
  // The expert tables, like the weights, are not written by the previous
  // kernel: their loads are issued now and stay in flight through the
  // router phase; the values go to shared memory just before the routing
  // decision reads them (E <= kMaxExperts <= kFThreads).
  const uint8_t* my_tab_g = threadIdx.x < E ? gu_tab[threadIdx.x] : nullptr;
  const uint8_t* my_tab_d = threadIdx.x < E ? dn_tab[threadIdx.x] : nullptr;
  // Router weights do not depend on the previous kernel: warm L2 with this
  // CTA's slices while that kernel finishes.
  if (threadIdx.x == 0)
    for (int t = c; t < T; t += G) {
      const int e = t / split, p = t - e * split;
      const int c0 = p * cs, c1 = min(nch, c0 + cs);
      if (c1 > c0) bulk_prefetch_l2(wr + ((size_t)e * nch + c0) * 8, uint32_t((c1 - c0) * 16));
    }
  __syncthreads();
  pdl_allow_next_grid();
  pdl_wait_prior_grid();  // x comes from the previous kernel
  // Counter 1 only grows, by G per call: the call's target is the next
  // multiple of G.  Read after the wait, so that the previous call on this
  // workspace is complete; no CTA of this call adds to it before every CTA
  // has read it (adds come after the routing decision, which needs every
  // CTA's router partials).
  uint64_t tgt1 = 0;
  if (threadIdx.x == 0) {
    const uint64_t b1 = ld_acquire_u64(&cnt[1]);
    tgt1 = b1 - b1 % uint64_t(G) + uint64_t(G);
  }

  // ---- phase A: router partials, written to every CTA's replica ----------
  const uint4* x4 = reinterpret_cast<const uint4*>(x);
  const uint4* w4 = reinterpret_cast<const uint4*>(wr);
  for (int t = c; t < T; t += G) {
    const int e = t / split, p = t - e * split;
    const int c0 = p * cs, c1 = min(nch, c0 + cs);
    float s = 0.f, cc = 0.f;
    for (int ch = c0 + threadIdx.x; ch < c1; ch += kFThreads) {
      const uint4 a = __ldcg(x4 + ch);
      const uint4 b = __ldcs(w4 + (size_t)e * nch + ch);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
      const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // bf16 x bf16 has at most 16 significant bits: exact in fp32
        comp_add(s, cc, __fmul_rn(bf16_bits_to_f32(aw[q] & 0xFFFFu), bf16_bits_to_f32(bw[q] & 0xFFFFu)));
        comp_add(s, cc, __fmul_rn(bf16_bits_to_f32(aw[q] >> 16), bf16_bits_to_f32(bw[q] >> 16)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      const float c2 = __shfl_xor_sync(0xffffffffu, cc, o);
      comp_merge(s, cc, s2, c2);
    }
    if (lane == 0) {
      red_s[warp] = s;
      red_c[warp] = cc;
    }
    __syncthreads();
    // warps past the task's chunks hold (0, 0), which a merge leaves as is
    const int wused = min(kFWarps, (c1 - c0 + 31) >> 5);
    float ts = red_s[0], tc = red_c[0];
    for (int w = 1; w < wused; ++w) comp_merge(ts, tc, red_s[w], red_c[w]);
    // one copy per CTA, so that no L2 line is read by every SM below
    const float2 pv = make_float2(nonzero_bits(ts), nonzero_bits(tc));
    for (int r = threadIdx.x; r < G; r += kFThreads) st_relaxed_f2(part + (size_t)r * T + t, pv);
    __syncthreads();
  }

  // x -> f16 (one power-of-two prescale) while the other CTAs finish phase A
  uint4 xr[kMaxXChunksPerThread];
  float mx = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxXChunksPerThread; ++i) {
    const int ch = threadIdx.x + i * kFThreads;
    xr[i] = ch < nch ? __ldcg(x4 + ch) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t vw[4] = {xr[i].x, xr[i].y, xr[i].z, xr[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      mx = fmaxf(mx, fmaxf(fabsf(bf16_bits_to_f32(vw[e] & 0xFFFFu)),
                           fabsf(bf16_bits_to_f32(vw[e] >> 16))));
  }
  mx = warp_max(mx);
  if (lane == 0) red_s[warp] = mx;
  __syncthreads();
  float gmax = red_s[0];
#pragma unroll
  for (int w = 1; w < kFWarps; ++w) gmax = fmaxf(gmax, red_s[w]);
  const int sx = min(f16_prescale_exponent(gmax), 127);
  const float two_s = scalbnf(1.0f, sx);
  const float inv = scalbnf(1.0f, -sx);
#pragma unroll
  for (int i = 0; i < kMaxXChunksPerThread; ++i) {
    const int ch = threadIdx.x + i * kFThreads;
    if (ch < nch) {
      const uint4 v = xr[i];
      uint4 o;
      o.x = pack_f16x2_scaled(bf16_bits_to_f32(v.x & 0xFFFFu), bf16_bits_to_f32(v.x >> 16), two_s);
      o.y = pack_f16x2_scaled(bf16_bits_to_f32(v.y & 0xFFFFu), bf16_bits_to_f32(v.y >> 16), two_s);
      o.z = pack_f16x2_scaled(bf16_bits_to_f32(v.z & 0xFFFFu), bf16_bits_to_f32(v.z >> 16), two_s);
      o.w = pack_f16x2_scaled(bf16_bits_to_f32(v.w & 0xFFFFu), bf16_bits_to_f32(v.w >> 16), two_s);
      xs[(ch & 3) * Lg.nblk + (ch >> 2)] = o;  // chunk q = ch % 4 of block ch / 4
    }
  }

  if (threadIdx.x < E) {
    tab_g[threadIdx.x] = my_tab_g;
    tab_d[threadIdx.x] = my_tab_d;
  }  // read after the __syncthreads that ends the routing decision

  // ---- routing decision (every CTA, same fixed-order fold) ---------------
  // Warp 0 polls this CTA's replica until every partial has arrived (the
  // values are their own signal: no separate counter and no second round
  // trip), folds them, and clears the replica for the next call.
  if (warp == 0) {
    float2* mine = part + (size_t)c * T;
    bool got = true;
    for (int e = lane; e < ((E + 31) & ~31); e += 32) {
      float lg = 0.f;
      if (e < E) {
        float2 v[kMaxRouterSplit];
        got = poll_partials(mine + (size_t)e * split, split, v) && got;
#pragma unroll
        for (int p = 0; p < kMaxRouterSplit; ++p)
          if (p < split) st_relaxed_f2(mine + (size_t)e * split + p, make_float2(0.f, 0.f));
        float s = v[0].x, cc = v[0].y;
#pragma unroll
        for (int p = 1; p < kMaxRouterSplit; ++p)
          if (p < split) comp_merge(s, cc, v[p].x, v[p].y);
        lg = __fadd_rn(s, cc);
        slog[e] = lg;
      }
      if (E <= 32) warp_topk_softmax32(lg, E, top_k, lane, sidx, sprob);
    }
    if (E > 32) {
      __syncwarp();
      warp_topk_softmax(slog, E, top_k, lane, sidx, sprob);
    }
    got = __all_sync(0xffffffffu, got);
    if (lane == 0) *sflag = got ? 1 : 0;
  }
  __syncthreads();
  if (*sflag == 0) {  // nothing of ours is in flight yet
    if (threadIdx.x == 0) flag_error(err, kErrTimeout);
    return;
  }
  // The selected experts' buffers must be usable by the bulk copies: a null
  // or misaligned pointer is reported (every CTA decides alike) and nothing
  // is copied from it.
  {
    int bad = 0;
    for (int j = 0; j < top_k; ++j) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(tab_g[sidx[j]]);
      const uintptr_t b = reinterpret_cast<uintptr_t>(tab_d[sidx[j]]);
      if (a == 0 || b == 0) bad = bad ? bad : kErrNull;
      else if ((a | b) & 15u) bad = bad ? bad : kErrAlign;
    }
    if (bad) {
      if (threadIdx.x == 0) flag_error(err, bad);
      return;
    }
  }
  if (c == 0 && threadIdx.x < top_k) {
    out_idx[threadIdx.x] = sidx[threadIdx.x];
    out_prob[threadIdx.x] = sprob[threadIdx.x];
  }

  // ---- phases B + C ----------------------------------------------------------
  const int nitems_d = nhb * P.nchunk;  // down item k = (chunk k / nhb, slice k % nhb)
  const int nq = nhb * 16;              // this CTA's gate/up records
  const int nit = nq > warp ? (nq - warp + kFWarps - 1) / kFWarps : 0;
  uint8_t* wbase = gring + (size_t)warp * P.gslots * Lg.bytes;
  uint64_t* wbars = gbars + warp * kMaxGuSlots;
  // next record to request: (expert j_iss, row r_iss), advanced by kFWarps
  // records per request without a division
  int j_iss = (qa + warp) / inter, r_iss = (qa + warp) - j_iss * inter;
  auto issue_gu = [&](int sl) {  // lane 0: the next record of this warp -> slot sl
    const int j = j_iss, r = r_iss;
    r_iss += kFWarps;
    if (r_iss >= inter) {
      r_iss -= inter;
      ++j_iss;
    }
    const uint32_t bar = smem_u32(&wbars[sl]);
    mbar_arrive_expect_tx(bar, uint32_t(Lg.bytes));
    bulk_g2s(smem_u32(wbase + (size_t)sl * Lg.bytes),
             tab_g[sidx[j]] + (int64_t)r * Lg.bytes, uint32_t(Lg.bytes),
             bar, policy);
  };
  auto issue_dn = [&](int k) {  // one thread: down item k -> slot k % dslots
    const int ch = k / nhb, i = k - ch * nhb;
    const int g = hb0 + i, j = g / spe, sl = g - j * spe;
    const int r0 = ch * rc, nr = min(rc, hidden - r0);
    const int s = k % P.dslots;
    const uint32_t bar = smem_u32(&dbars[s]);
    uint8_t* dst = dring + (size_t)s * P.item;
    const uint8_t* src = tab_d[sidx[j]];
    mbar_arrive_expect_tx(bar, uint32_t(nr * 9));
    bulk_g2s(smem_u32(dst), src + Ld.code_at(sl, r0), uint32_t(nr * 8), bar, policy);
    bulk_g2s(smem_u32(dst + (size_t)rc * 8), src + Ld.scale_at(sl >> 1, r0), uint32_t(nr), bar,
             policy);
  };
  if (lane == 0)
    for (int t = 0; t < min(P.gslots, nit); ++t) issue_gu(t);  // item t -> slot t
  if (threadIdx.x == 32) {
    const int n0 = min(P.dslots, nitems_d);
    for (int k = 0; k < n0; ++k) issue_dn(k);
    *d_issued = n0;
  }
  __syncthreads();  // d_issued visible before any warp may refill

  float acc[kRowsPerThread];
#pragma unroll
  for (int m = 0; m < kRowsPerThread; ++m) acc[m] = 0.f;
  // this warp's next down item kd = (chunk kd_ch, slice kd_i), in slot kd_s
  // with mbarrier parity kd_ph, on its kd_pass-th use of that slot
  int kd = 0, kd_ch = 0, kd_i = 0, kd_s = 0, kd_pass = 0;
  uint32_t kd_ph = 0;
  // Down item kd for this thread's rows (t + 512 m of the item's row chunk);
  // the last of the 16 warps to finish a slot refills it.
  auto do_down = [&]() {
    const int ch = kd_ch, i = kd_i;
    const int r0 = kOneChunk ? 0 : ch * rc, nr = kOneChunk ? KH : min(rc, hidden - r0);
    const int s = kd_s;
    const uint8_t* slot = dring + (size_t)s * P.item;
    float hv[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 t4 = reinterpret_cast<const float4*>(hs + i * 16)[q];
      hv[4 * q + 0] = t4.x;
      hv[4 * q + 1] = t4.y;
      hv[4 * q + 2] = t4.z;
      hv[4 * q + 3] = t4.w;
    }
    const float pj = sprob[(hb0 + i) / spe];
#pragma unroll
    for (int m = 0; m < kRowsPerThread; ++m) {
      const int r = threadIdx.x + m * kFThreads;  // row within the chunk
      if (r < nr) {
        const uint2 cw = *reinterpret_cast<const uint2*>(slot + (size_t)r * 8);
        const float ps = pj * e8m0_to_f32(slot[(size_t)rc * 8 + r]);  // exact
        acc[m] = fmaf(ps, dot16_f32(cw, hv), acc[m]);
      }
    }
    if (i == nhb - 1) {  // last slice of this row chunk: publish the partial sums
#pragma unroll
      for (int m = 0; m < kRowsPerThread; ++m) {
        const int r = threadIdx.x + m * kFThreads;
        if (r < nr) opart[(size_t)c * hidden + r0 + r] = acc[m];
        acc[m] = 0.f;
      }
    }
    __syncwarp();
    // dcons[s] only grows: the consumers of the p-th item in slot s draw
    // 16 p .. 16 p + 15, and the one that draws the last value refills it
    if (lane == 0 && atomicAdd(&dcons[s], 1) == kFWarps * kd_pass + kFWarps - 1) {
      const int nk = kd + P.dslots;
      if (nk < nitems_d) {
        issue_dn(nk);
        atomicMax(d_issued, nk + 1);
      }
    }
    ++kd;
    if (++kd_i == nhb) {
      kd_i = 0;
      ++kd_ch;
    }
    if (++kd_s == P.dslots) {
      kd_s = 0;
      ++kd_pass;
      kd_ph ^= 1u;
    }
  };
  auto down_ready = [&]() -> bool {  // warp-uniform, non-blocking
    bool ok = mbar_test_wait(smem_u32(&hbars[kd_i]), 0u) &&
              mbar_test_wait(smem_u32(&dbars[kd_s]), kd_ph);
    return __all_sync(0xffffffffu, ok);
  };

  bool failed = false;
  int t = 0, sl = 0;  // record t of this warp sits in ring slot sl with parity gph
  uint32_t gph = 0;
  for (; t < nit; ++t) {
    const bool ok = mbar_wait_sleep_bounded(smem_u32(&wbars[sl]), gph, 256u);
    if (!__all_sync(0xffffffffu, ok)) {
      failed = true;
      break;
    }
    const uint8_t* rec = wbase + (size_t)sl * Lg.bytes;
    float ag = 0.f, au = 0.f;
#pragma unroll
    for (int ib = 0; ib < NBG; ++ib) {
      const int b = 32 * ib + lane;
      if (b < Lg.nblk) {
        uint32_t xv[16];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const uint4 tq = xs[qq * Lg.nblk + b];
          xv[4 * qq + 0] = tq.x;
          xv[4 * qq + 1] = tq.y;
          xv[4 * qq + 2] = tq.z;
          xv[4 * qq + 3] = tq.w;
        }
        const uint4 cg = *reinterpret_cast<const uint4*>(rec + Lg.gate_codes() + b * 16);
        const uint4 cu = *reinterpret_cast<const uint4*>(rec + Lg.up_codes() + b * 16);
        ag = fmaf(dot32(cg, xv), e8m0_to_f32(rec[Lg.gate_scales() + b]), ag);
        au = fmaf(dot32(cu, xv), e8m0_to_f32(rec[Lg.up_scales() + b]), au);
      }
    }
    const float pg = *reinterpret_cast<const float*>(rec + Lg.post);
    const float pu = *reinterpret_cast<const float*>(rec + Lg.post + 4);
    __syncwarp();
    if (lane == 0 && t + P.gslots < nit) issue_gu(sl);  // record t + gslots into this slot
    if (++sl == P.gslots) {
      sl = 0;
      gph ^= 1u;
    }
    const float v = warp_sum2(ag, au, lane);  // lanes 0-15: g, 16-31: u
    const float g = __shfl_sync(0xffffffffu, v, 0) * inv * pg;
    const float u = __shfl_sync(0xffffffffu, v, 16) * inv * pu;
    if (lane == 0) {
      const int r = warp + t * kFWarps;  // record index within the CTA
      hs[r] = silu_mul(g, u);
      mbar_arrive(smem_u32(&hbars[r >> 4]));  // releases hs[r] to every warp
    }
    while (kd < nitems_d && down_ready()) do_down();  // fill the wait with down work
  }
  if (failed) {  // timed out at record t: let this warp's issued records land
    if (lane == 0) {
      const int issued = min(nit, t + P.gslots);
      for (int u = t + 1; u < issued; ++u)
        (void)mbar_wait_bounded(smem_u32(&wbars[u % P.gslots]), uint32_t((u / P.gslots) & 1));
      *sfail = 1;
    }
  } else {
    // the remaining slices, waiting for them (bounded)
    while (kd < nitems_d) {
      bool ok = mbar_wait_sleep_bounded(smem_u32(&hbars[kd_i]), 0u, 256u);
      ok = ok && mbar_wait_sleep_bounded(smem_u32(&dbars[kd_s]), kd_ph, 256u);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) *sfail = 1;
        break;
      }
      do_down();
    }
  }
  __syncthreads();
  if (*sfail) {
    if (threadIdx.x == 0) {
      flag_error(err, kErrTimeout);
      const int issued = *d_issued;  // let the issued down items land
      for (int k = max(0, issued - P.dslots); k < issued; ++k)
        (void)mbar_wait_bounded(smem_u32(&dbars[k % P.dslots]), uint32_t((k / P.dslots) & 1));
    }
    return;
  }
  if (nhb == 0) {  // no slices: publish zeros, so that phase D reads every CTA
    for (int r = threadIdx.x; r < hidden; r += kFThreads) opart[(size_t)c * hidden + r] = 0.f;
    __syncthreads();
  }

  // ---- phase D: fixed-order sum of the partial vectors of our rows -------
  if (threadIdx.x == 0) {
    red_release_add(&cnt[1], 1u);  // after the CTA's partial-vector writes
    *sflag = wait_counter(&cnt[1], tgt1) ? 1 : 0;
  }
  __syncthreads();
  if (*sflag == 0) {
    if (threadIdx.x == 0) flag_error(err, kErrTimeout);
    return;
  }
  const int o0 = int((int64_t)hidden * c / G), o1 = int((int64_t)hidden * (c + 1) / G);
  const int nro = o1 - o0;
  float* gat = reinterpret_cast<float*>(dring);  // [G][nro]; both rings are free
  // all loads of a thread are issued before the first is used: one L2 round
  // trip per batch of kGatherBatch, not one per element
  constexpr int kGatherBatch = 8;
  for (int base = 0; base < G * nro; base += kFThreads * kGatherBatch) {
    float v[kGatherBatch];
#pragma unroll
    for (int u = 0; u < kGatherBatch; ++u) {
      const int idx = base + threadIdx.x + u * kFThreads;
      const int cc = idx / nro, rr = idx - cc * nro;
      v[u] = idx < G * nro ? __ldcg(opart + (size_t)cc * hidden + o0 + rr) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kGatherBatch; ++u) {
      const int idx = base + threadIdx.x + u * kFThreads;
      if (idx < G * nro) gat[idx] = v[u];
    }
  }
  __syncthreads();
  for (int rr = warp; rr < nro; rr += kFWarps) {
    float sum = 0.f;
    for (int cc = lane; cc < G; cc += 32) sum += gat[cc * nro + rr];
    sum = warp_sum(sum);
    if (lane == 0) out[o0 + rr] = f32_to_bf16_rne(sum);
  }

}

std::atomic<int> g_coop_pdl_state{0};  // 0 unknown, 1 cooperative + PDL accepted, 2 refused

}  // namespace

size_t moe_fused_workspace_bytes(int64_t hidden) {
  return size_t(kWsHOffset) + size_t(kMaxMoeGrid) * size_t(hidden) * 4;
}

cudaError_t launch_moe_fused(const uint16_t* x, int hidden, int inter, const uint16_t* wr, int E,
                             int top_k, const uint8_t* const* gu, const uint8_t* const* dn,
                             uint16_t* out,
                             int32_t* out_idx, float* out_prob, void* ws, cudaStream_t s,
                             bool pdl) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorNoDevice;
  const int grid = di->sms < kMaxMoeGrid ? di->sms : kMaxMoeGrid;
  if (hidden > kFThreads * kMaxXChunksPerThread * 8) return cudaErrorInvalidConfiguration;
  MoePlan plan;
  if (!make_plan(hidden, inter, top_k, grid, di->smem_optin, plan))
    return cudaErrorInvalidConfiguration;
  int split = grid / E;
  if (split < 1) split = 1;
  if (split > kMaxRouterSplit) split = kMaxRouterSplit;

  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t r =
        ensure_smem(*di, kern, plan.total);
    if (r != cudaSuccess) return r;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = plan.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // The first launch finds out whether the runtime takes both attributes
    // together; a refused launch inside a stream capture could invalidate the
    // capture, so that first try never happens while capturing.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (g_coop_pdl_state == 0 && cudaStreamIsCapturing(s, &cap) != cudaSuccess)
      return cudaErrorUnknown;
    const bool try_pdl = pdl && (g_coop_pdl_state == 1 ||
                                 (g_coop_pdl_state == 0 && cap == cudaStreamCaptureStatusNone));
    cfg.numAttrs = try_pdl ? 2 : 1;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    r = cudaLaunchKernelEx(&cfg, kern, x, hidden, inter, wr, E, top_k, gu, dn, out, out_idx,
                           out_prob, wsb, split, plan, di->error_word);
    if (try_pdl) {
      if (r == cudaSuccess) {
        g_coop_pdl_state = 1;
      } else if (g_coop_pdl_state == 0) {
        // this runtime does not combine the two attributes: cooperative only
        (void)cudaGetLastError();
        g_coop_pdl_state = 2;
        cfg.numAttrs = 1;
        r = cudaLaunchKernelEx(&cfg, kern, x, hidden, inter, wr, E, top_k, gu, dn, out, out_idx,
                               out_prob, wsb, split, plan, di->error_word);
      }
    }
    return r;
  };
  // gpt-oss-20b's expert shape gets a kernel with the sizes fixed
  if (hidden == 2880 && inter == 2880 && plan.rc == hidden)
    return go(moe_fused_kernel<3, 2880, 2880>);
  switch ((hidden / 32 + 31) / 32) {
#define TT_FU(nb) \
  case nb: return go(moe_fused_kernel<nb, 0, 0>);
    TT_FU(1) TT_FU(2) TT_FU(3) TT_FU(4) TT_FU(5) TT_FU(6) TT_FU(7) TT_FU(8)
#undef TT_FU
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tt
