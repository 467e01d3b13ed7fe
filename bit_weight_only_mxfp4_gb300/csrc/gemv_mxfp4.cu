// CUDA-core MXFP4 gate/up SwiGLU matvec for small batches (m = 1..8).
//
// Method: ThinTensor devlog (kerbin.cskartikey.dev/@satvikhardat), Dev Log #4
// "Where Blackwell helps": read the MXFP4 bytes, use the block scales,
// multiply against bf16 activations, accumulate safely, then apply the row
// postscale; the gate/up pair feeds the gated activation of Dev Log #2.
// Decode is a weight-read problem (Dev Log #4, "Why gate/up was the right
// target"), so the kernel is built to stream the packed codes once at HBM
// speed:
//
//  * persistent grid, one CTA per SM, each CTA owning a contiguous range of
//    row records of the packed layout (layout.cuh);
//  * every warp runs its own ring of `slots` shared-memory slots, refilled
//    by one-instruction bulk copies (TMA, non-tensor) signalled on an
//    mbarrier; the first copies are issued before the programmatic-
//    dependent-launch wait, so weight streaming overlaps the previous
//    kernel's tail;
//  * lane l owns the 32-weight blocks l, l+32, l+64, ... of every row, so
//    its slice of x is converted once (to f16 after an exact power-of-two
//    prescale) and reused for every row;
//  * E2M1 pairs are widened with cvt.rn.f16x2.e2m1x2 and multiplied into
//    fp32 with fma.rn.f32.f16 (the e2m1 x f16 products are exact), the
//    block's E8M0 scale is applied once per 32 products, and the split-K
//    partial sums meet in a warp-shuffle reduction;
//  * K is always looped in bounded 1024-wide chunks (the project page's
//    wide-matvec devlog: never pad K into one oversized tile).
#include "common.cuh"
#include "launch.h"
#include "layout.cuh"
#include "mxfp4_core.cuh"

namespace tt {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

// Launch shape of the m = 1 kernel for k <= 3072 (x fits in 128 registers):
// CTAs per SM, ring slots per warp and records per bulk copy.
#ifndef TT_M1_CTAS_PER_SM
#define TT_M1_CTAS_PER_SM 2
#endif
#ifndef TT_M1_SLOTS
#define TT_M1_SLOTS 2
#endif
#ifndef TT_M1_RPC
#define TT_M1_RPC 1
#endif
// When the register-x and shared-x kernels allow the dependent launch:
// 0 = at entry (measured best), 1 = once x has been read.
#ifndef TT_M1_LATE_TRIGGER
#define TT_M1_LATE_TRIGGER 0
#endif
// Each CTA prefetches its whole weight range into L2 at launch, so that the
// number of bytes in flight is not limited by the shared-memory ring.
#ifndef TT_M1_L2PF
#define TT_M1_L2PF 0
#endif
// m = 1 with x staged in shared memory (1) or held in registers (0), and the
// warps per CTA of the shared-memory variant.
#ifndef TT_M1_XSMEM
#define TT_M1_XSMEM 1
#endif
// m = 1 through the stage-pipelined, warp-specialised kernel (and its ring
// depth cap).
#ifndef TT_M1_STAGED
#define TT_M1_STAGED 0
#endif
#ifndef TT_M1X_CTAS_PER_SM
#define TT_M1X_CTAS_PER_SM 1
#endif
#ifndef TT_M1S_SLOTS
#define TT_M1S_SLOTS 8
#endif
#ifndef TT_M1S_INTERLEAVE
#define TT_M1S_INTERLEAVE 0
#endif
// When the dependent launch is allowed: 0 = at entry, 1 = once the producer
// has issued the last copy of this kernel.
#ifndef TT_M1S_TRIGGER
#define TT_M1S_TRIGGER 1
#endif
// Queue the stages beyond the ring into L2 at entry.
#ifndef TT_M1S_L2PF
#define TT_M1S_L2PF 1
#endif
#ifndef TT_M1_WARPS
#define TT_M1_WARPS 16
#endif


// ---------------------------------------------------------------------------
// m = 1, x held in registers.  NB = number of 1024-wide K chunks
// (k <= 1024*NB); RPC = records per bulk copy (1 or 2).
// ---------------------------------------------------------------------------
template <int NB, int RPC>
__global__ void __launch_bounds__(kThreads, (NB <= 3 ? 2 : 1))
    swiglu_mxfp4_m1_kernel(const uint8_t* __restrict__ packed, int n, int k,
                           const uint16_t* __restrict__ x, uint16_t* __restrict__ h, int slots,
                           int32_t* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SwigluRecord L(k);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r0 = int((int64_t)n * blockIdx.x / gridDim.x);
  const int r1 = int((int64_t)n * (blockIdx.x + 1) / gridDim.x);
  const int units = (r1 - r0 + RPC - 1) / RPC;
  const int nitems = units > warp ? (units - warp + kWarps - 1) / kWarps : 0;

  WarpRing ring;
  ring.slots = slots;
  ring.rec_bytes = L.bytes;
  ring.slot_bytes = RPC * L.bytes;
  ring.base = smem + (size_t)warp * slots * ring.slot_bytes;
  ring.bars = reinterpret_cast<uint64_t*>(smem + (size_t)kWarps * slots * ring.slot_bytes) +
              warp * slots;
  ring.packed = packed;
  ring.policy = l2_evict_first_policy();
  ring.init(lane);

  auto first_of = [&](int j) { return r0 + (warp + j * kWarps) * RPC; };
  auto count_of = [&](int first) { return min(RPC, r1 - first); };

  if (!TT_M1_LATE_TRIGGER) pdl_allow_next_grid();
  // Weights do not depend on the previous kernel: start streaming them now.
  if (lane == 0)
    for (int j = 0; j < min(slots, nitems); ++j) ring.issue_to(j, first_of(j), count_of(first_of(j)));
  pdl_wait_prior_grid();

  // x is read from global memory once per CTA (not once per warp: thousands
  // of warps fetching the same few lines would queue on a few L2 slices).
  uint4* xs = reinterpret_cast<uint4*>(
      smem + (size_t)kWarps * slots * ring.slot_bytes + (size_t)kWarps * slots * 8);
  for (int c = threadIdx.x; c < (k >> 3); c += kThreads)
    xs[c] = reinterpret_cast<const uint4*>(x)[c];
  __syncthreads();

  // x slice of this lane -> f16x2 registers, prescaled by 2^sx (exact).
  uint32_t xr[NB][16];
  float xmax = 0.f;
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    const int b = 32 * i + lane;
    uint4 q[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                  make_uint4(0, 0, 0, 0)};
    if (b < L.nblk) {
#pragma unroll
      for (int t = 0; t < 4; ++t) q[t] = xs[b * 4 + t];
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      xr[i][4 * t + 0] = q[t].x;
      xr[i][4 * t + 1] = q[t].y;
      xr[i][4 * t + 2] = q[t].z;
      xr[i][4 * t + 3] = q[t].w;
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      xmax = fmaxf(xmax, fabsf(bf16_bits_to_f32(xr[i][t] & 0xFFFFu)));
      xmax = fmaxf(xmax, fabsf(bf16_bits_to_f32(xr[i][t] >> 16)));
    }
  }
  xmax = warp_max(xmax);
  const int sx = min(f16_prescale_exponent(xmax), 127);
  const float two_s = scalbnf(1.0f, sx);
#pragma unroll
  for (int i = 0; i < NB; ++i)
#pragma unroll
    for (int t = 0; t < 16; ++t)
      xr[i][t] = pack_f16x2_scaled(bf16_bits_to_f32(xr[i][t] & 0xFFFFu),
                                   bf16_bits_to_f32(xr[i][t] >> 16), two_s);
  if (TT_M1_LATE_TRIGGER) pdl_allow_next_grid();
  const float inv = scalbnf(1.0f, -sx);  // exact power of two
  EpilogueBatch ep;

  for (int j = 0; j < nitems; ++j) {
    const uint8_t* slot = ring.wait_next();
    if (slot == nullptr) {
      if (lane == 0) flag_error(err, kErrTimeout);
      ring.drain(j, nitems);
      return;
    }
    const int first = first_of(j);
    const int count = count_of(first);
    float ag[RPC], au[RPC], pg[RPC], pu[RPC];
#pragma unroll
    for (int rr = 0; rr < RPC; ++rr) {
      ag[rr] = au[rr] = 0.f;
      pg[rr] = pu[rr] = 1.f;
      if (rr < count) {
        const uint8_t* rec = slot + rr * L.bytes;
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          const int b = 32 * i + lane;
          if (b < L.nblk) {
            const uint4 cg = *reinterpret_cast<const uint4*>(rec + L.gate_codes() + b * 16);
            const uint4 cu = *reinterpret_cast<const uint4*>(rec + L.up_codes() + b * 16);
            const float sg = e8m0_to_f32(rec[L.gate_scales() + b]);
            const float su = e8m0_to_f32(rec[L.up_scales() + b]);
            ag[rr] = fmaf(dot32(cg, xr[i]), sg, ag[rr]);
            au[rr] = fmaf(dot32(cu, xr[i]), su, au[rr]);
          }
        }
        pg[rr] = *reinterpret_cast<const float*>(rec + L.post);
        pu[rr] = *reinterpret_cast<const float*>(rec + L.post + 4);
      }
    }
    __syncwarp();
    if (lane == 0 && j + slots < nitems) {
      const int f = first_of(j + slots);
      ring.issue_to(ring.cur, f, count_of(f));  // the slot just consumed
    }
    ring.advance();
    if constexpr (RPC == 2) {
      // lanes 0-7: g0, 8-15: u0, 16-23: g1, 24-31: u1
      const float v = warp_sum4(ag[0], au[0], ag[1], au[1], lane);
      if (ep.fill > 30) ep.flush(h);
      ep.put(v, 0, 8, pg[0], pu[0], inv, first, lane);
      if (count > 1) ep.put(v, 16, 24, pg[1], pu[1], inv, first + 1, lane);
    } else {
      const float v = warp_sum2(ag[0], au[0], lane);  // lanes 0-15: g, 16-31: u
      if (ep.fill > 31) ep.flush(h);
      ep.put(v, 0, 16, pg[0], pu[0], inv, first, lane);
    }
  }
  ep.flush(h);
}

// ---------------------------------------------------------------------------
// m = 1, x staged once per CTA in shared memory as f16 (prescaled by 2^sx),
// laid out chunk-major: 16-byte chunk q (0..3) of block b at xs[q*nblk + b],
// so a warp reading blocks b..b+31 touches 32 consecutive 16-byte words.
// Keeping x out of registers lets WARPS warps per CTA stay resident while
// the next kernel's CTA (programmatic dependent launch) shares the SM.
// NB = number of 1024-wide K chunks; RPC = records per bulk copy.
// ---------------------------------------------------------------------------
template <int NB, int RPC, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 2)
    swiglu_mxfp4_m1x_kernel(const uint8_t* __restrict__ packed, int n, int k,
                            const uint16_t* __restrict__ x, uint16_t* __restrict__ h, int slots,
                            int32_t* err) {
  constexpr int THREADS = WARPS * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const SwigluRecord L(k);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r0 = int((int64_t)n * blockIdx.x / gridDim.x);
  const int r1 = int((int64_t)n * (blockIdx.x + 1) / gridDim.x);
  const int units = (r1 - r0 + RPC - 1) / RPC;
  const int nitems = units > warp ? (units - warp + WARPS - 1) / WARPS : 0;

  const size_t ring_bytes = (size_t)WARPS * slots * RPC * L.bytes;
  WarpRing ring;
  ring.slots = slots;
  ring.rec_bytes = L.bytes;
  ring.slot_bytes = RPC * L.bytes;
  ring.base = smem + (size_t)warp * slots * ring.slot_bytes;
  ring.bars = reinterpret_cast<uint64_t*>(smem + ring_bytes) + warp * slots;
  ring.packed = packed;
  ring.policy = l2_evict_first_policy();
  uint4* xraw = reinterpret_cast<uint4*>(smem + ring_bytes + (size_t)WARPS * slots * 8);
  uint4* xs = xraw + (k >> 3);
  float* red = reinterpret_cast<float*>(xs + (k >> 3));
  ring.init(lane);

  auto first_of = [&](int j) { return r0 + (warp + j * WARPS) * RPC; };
  auto count_of = [&](int first) { return min(RPC, r1 - first); };

  if (!TT_M1_LATE_TRIGGER) pdl_allow_next_grid();
  if (TT_M1_L2PF) {
    // The CTA's records are contiguous: ask L2 for all of them now, in
    // 16 KB pieces spread over the CTA's threads.
    const char* base = reinterpret_cast<const char*>(packed) + (int64_t)r0 * L.bytes;
    const int64_t total = (int64_t)(r1 - r0) * L.bytes;
    constexpr int64_t kPiece = 16384;
    for (int64_t off = (int64_t)threadIdx.x * kPiece; off < total; off += (int64_t)THREADS * kPiece)
      bulk_prefetch_l2(base + off, uint32_t(min(kPiece, total - off)));
  }
  // Weights do not depend on the previous kernel: start streaming them now.
  if (lane == 0)
    for (int j = 0; j < min(slots, nitems); ++j) ring.issue_to(j, first_of(j), count_of(first_of(j)));
  pdl_wait_prior_grid();

  // x: one global read per CTA, CTA-wide max |x| -> exact power-of-two
  // prescale, then f16 in the chunk-major layout.
  const int nchunk16 = k >> 3;
  float mx = 0.f;
  const uint64_t x_policy = l2_evict_last_policy();
  for (int c = threadIdx.x; c < nchunk16; c += THREADS) {
    const uint4 v = ld_global_v4_hint(reinterpret_cast<const uint4*>(x) + c, x_policy);
    xraw[c] = v;
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(bf16_bits_to_f32(v.x & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.x >> 16))),
                         fmaxf(fabsf(bf16_bits_to_f32(v.y & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.y >> 16)))));
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(bf16_bits_to_f32(v.z & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.z >> 16))),
                         fmaxf(fabsf(bf16_bits_to_f32(v.w & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.w >> 16)))));
  }
  mx = warp_max(mx);
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  float gmax = red[0];
#pragma unroll
  for (int w = 1; w < WARPS; ++w) gmax = fmaxf(gmax, red[w]);
  const int sx = min(f16_prescale_exponent(gmax), 127);
  const float two_s = scalbnf(1.0f, sx);
  for (int c = threadIdx.x; c < nchunk16; c += THREADS) {
    const uint4 v = xraw[c];
    uint4 o;
    o.x = pack_f16x2_scaled(bf16_bits_to_f32(v.x & 0xFFFFu), bf16_bits_to_f32(v.x >> 16), two_s);
    o.y = pack_f16x2_scaled(bf16_bits_to_f32(v.y & 0xFFFFu), bf16_bits_to_f32(v.y >> 16), two_s);
    o.z = pack_f16x2_scaled(bf16_bits_to_f32(v.z & 0xFFFFu), bf16_bits_to_f32(v.z >> 16), two_s);
    o.w = pack_f16x2_scaled(bf16_bits_to_f32(v.w & 0xFFFFu), bf16_bits_to_f32(v.w >> 16), two_s);
    xs[(c & 3) * L.nblk + (c >> 2)] = o;  // chunk q = c % 4 of block b = c / 4
  }
  __syncthreads();
  if (TT_M1_LATE_TRIGGER) pdl_allow_next_grid();
  const float inv = scalbnf(1.0f, -sx);  // exact power of two
  EpilogueBatch ep;

  for (int j = 0; j < nitems; ++j) {
    const uint8_t* slot = ring.wait_next();
    if (slot == nullptr) {
      if (lane == 0) flag_error(err, kErrTimeout);
      ring.drain(j, nitems);
      return;
    }
    const int first = first_of(j);
    const int count = count_of(first);
    float ag[RPC], au[RPC];
#pragma unroll
    for (int rr = 0; rr < RPC; ++rr) ag[rr] = au[rr] = 0.f;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int b = 32 * i + lane;
      if (b < L.nblk) {
        uint32_t xv[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 t = xs[q * L.nblk + b];
          xv[4 * q + 0] = t.x;
          xv[4 * q + 1] = t.y;
          xv[4 * q + 2] = t.z;
          xv[4 * q + 3] = t.w;
        }
#pragma unroll
        for (int rr = 0; rr < RPC; ++rr) {
          if (rr < count) {
            const uint8_t* rec = slot + rr * L.bytes;
            const uint4 cg = *reinterpret_cast<const uint4*>(rec + L.gate_codes() + b * 16);
            const uint4 cu = *reinterpret_cast<const uint4*>(rec + L.up_codes() + b * 16);
            const float sg = e8m0_to_f32(rec[L.gate_scales() + b]);
            const float su = e8m0_to_f32(rec[L.up_scales() + b]);
            ag[rr] = fmaf(dot32(cg, xv), sg, ag[rr]);
            au[rr] = fmaf(dot32(cu, xv), su, au[rr]);
          }
        }
      }
    }
    float pg[RPC], pu[RPC];
#pragma unroll
    for (int rr = 0; rr < RPC; ++rr) {
      const uint8_t* rec = slot + rr * L.bytes;
      pg[rr] = rr < count ? *reinterpret_cast<const float*>(rec + L.post) : 1.f;
      pu[rr] = rr < count ? *reinterpret_cast<const float*>(rec + L.post + 4) : 1.f;
    }
    __syncwarp();
    if (lane == 0 && j + slots < nitems) {
      const int f = first_of(j + slots);
      ring.issue_to(ring.cur, f, count_of(f));  // the slot just consumed
    }
    ring.advance();
    if constexpr (RPC == 2) {
      // lanes 0-7: g0, 8-15: u0, 16-23: g1, 24-31: u1
      const float v = warp_sum4(ag[0], au[0], ag[1], au[1], lane);
      if (ep.fill > 30) ep.flush(h);
      ep.put(v, 0, 8, pg[0], pu[0], inv, first, lane);
      if (count > 1) ep.put(v, 16, 24, pg[1], pu[1], inv, first + 1, lane);
    } else {
      const float v = warp_sum2(ag[0], au[0], lane);  // lanes 0-15: g, 16-31: u
      if (ep.fill > 31) ep.flush(h);
      ep.put(v, 0, 16, pg[0], pu[0], inv, first, lane);
    }
  }
  ep.flush(h);
}

// ---------------------------------------------------------------------------
// m = 1, stage-pipelined and warp-specialised.
//
// The CTA's records are consumed in stages of R consecutive records, each
// brought in by ONE bulk copy into a ring of `slots` shared-memory stages.
// Warp NB*R (the producer) issues the copies and, once every consumer warp
// has released a stage, runs the SwiGLU epilogue of its records and refills
// the slot.  Consumer warp w owns K chunk c = w % NB (lane l owns block
// 32c + l) of the stage's record w / NB, so it keeps only that 1024-wide
// slice of x (16 registers) and per stage does two 32-weight dot products,
// one warp reduction and one arrive: no per-record control flow.
// ---------------------------------------------------------------------------
template <int NB, int R>
__global__ void __launch_bounds__((NB * R + 1) * 32, 1)
    swiglu_mxfp4_m1s_kernel(const uint8_t* __restrict__ packed, int n, int k,
                            const uint16_t* __restrict__ x, uint16_t* __restrict__ h, int slots,
                            int32_t* err) {
  constexpr int W = NB * R;  // consumer warps
  extern __shared__ __align__(128) uint8_t smem[];
  const SwigluRecord L(k);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // Stage t of this CTA covers records [first(t), first(t) + cnt(t)).  With
  // TT_M1S_INTERLEAVE the CTAs take global stages round-robin, so the whole
  // grid sweeps the matrix front to back; otherwise each CTA owns a
  // contiguous range.
#if TT_M1S_INTERLEAVE
  const int nstage_all = (n + R - 1) / R;
  const int stages = nstage_all > (int)blockIdx.x
                         ? (nstage_all - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                         : 0;
  auto first = [&](int t) { return ((int)blockIdx.x + t * (int)gridDim.x) * R; };
  auto cnt = [&](int t) { return min(R, n - first(t)); };
#else
  const int r0 = int((int64_t)n * blockIdx.x / gridDim.x);
  const int r1 = int((int64_t)n * (blockIdx.x + 1) / gridDim.x);
  const int stages = (r1 - r0 + R - 1) / R;
  auto first = [&](int t) { return r0 + t * R; };
  auto cnt = [&](int t) { return min(R, r1 - (r0 + t * R)); };
#endif
  const int stage_bytes = R * L.bytes;
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)slots * stage_bytes);
  uint64_t* empty = full + slots;
  float* part = reinterpret_cast<float*>(empty + slots);  // [slots][R][NB][2]

  if (threadIdx.x == 0) {
    for (int s = 0; s < slots; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), W * 32);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (TT_M1S_TRIGGER == 0) pdl_allow_next_grid();

  if (warp == W) {
    // ---------------- producer and epilogue warp ----------------
    const uint64_t policy = l2_evict_first_policy();
    int issued = 0;
    auto issue = [&](int t) {  // lane 0 only
      const int s = t % slots;
      const uint32_t bytes = uint32_t(cnt(t) * L.bytes);
      mbar_arrive_expect_tx(smem_u32(&full[s]), bytes);
      bulk_g2s(smem_u32(ring + (size_t)s * stage_bytes), packed + (int64_t)first(t) * L.bytes,
               bytes, smem_u32(&full[s]), policy);
    };
    // Weights do not depend on the previous kernel: start streaming them now.
    if (lane == 0) {
      for (int t = 0; t < min(slots, stages); ++t) issue(t);
      // The stages that do not fit the ring yet: queue them into L2 now, so
      // their HBM reads happen while the ring drains.
      if (TT_M1S_L2PF)
        for (int t = slots; t < stages; ++t)
          bulk_prefetch_l2(packed + (int64_t)first(t) * L.bytes, uint32_t(cnt(t) * L.bytes));
    }
    issued = min(slots, stages);
    // Let the next kernel launch once every weight byte of this one has been
    // requested, so its prefetch queues behind this kernel's reads.
    if (TT_M1S_TRIGGER == 1 && stages <= slots) pdl_allow_next_grid();
    pdl_wait_prior_grid();  // h may still be read by the previous kernel
    for (int t = 0; t < stages; ++t) {
      const int s = t % slots;
      const bool ok = mbar_wait_bounded(smem_u32(&empty[s]), uint32_t((t / slots) & 1));
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) flag_error(err, kErrTimeout);
        // let the copies already issued land before the CTA may exit
        for (int u = t; u < issued; ++u)
          (void)mbar_wait_bounded(smem_u32(&full[u % slots]), uint32_t((u / slots) & 1));
        return;
      }
      if (lane < cnt(t)) {
        const float* p = part + ((size_t)s * R + lane) * NB * 2;
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int c = 0; c < NB; ++c) {
          g += p[2 * c];
          u += p[2 * c + 1];
        }
        const uint8_t* rec = ring + (size_t)s * stage_bytes + (size_t)lane * L.bytes;
        g *= *reinterpret_cast<const float*>(rec + L.post);
        u *= *reinterpret_cast<const float*>(rec + L.post + 4);
        h[first(t) + lane] = f32_to_bf16_rne(silu_mul(g, u));
      }
      __syncwarp();
      if (t + slots < stages) {
        if (lane == 0) issue(t + slots);
        ++issued;
        if (TT_M1S_TRIGGER == 1 && t + slots == stages - 1) pdl_allow_next_grid();
      }
    }
    return;
  }

  // ---------------- consumer warps ----------------
  const int chunk = warp % NB, rslot = warp / NB;
  const int b = 32 * chunk + lane;
  const bool active = b < L.nblk;
  pdl_wait_prior_grid();
  // This warp's slice of x -> f16x2, prescaled by a power of two chosen from
  // the slice's own max |x| (exact); partial sums are unscaled before they
  // meet the other chunks'.
  uint32_t xv[16];
  float xmax = 0.f;
  {
    const uint64_t xpol = l2_evict_last_policy();
    uint4 q[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                  make_uint4(0, 0, 0, 0)};
    if (active) {
      const uint4* src = reinterpret_cast<const uint4*>(x) + (size_t)b * 4;
#pragma unroll
      for (int t = 0; t < 4; ++t) q[t] = ld_global_v4_hint(src + t, xpol);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      xv[4 * t + 0] = q[t].x;
      xv[4 * t + 1] = q[t].y;
      xv[4 * t + 2] = q[t].z;
      xv[4 * t + 3] = q[t].w;
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      xmax = fmaxf(xmax, fabsf(bf16_bits_to_f32(xv[t] & 0xFFFFu)));
      xmax = fmaxf(xmax, fabsf(bf16_bits_to_f32(xv[t] >> 16)));
    }
  }
  xmax = warp_max(xmax);
  const int sx = min(f16_prescale_exponent(xmax), 127);
  const float two_s = scalbnf(1.0f, sx);
  const float inv = scalbnf(1.0f, -sx);
#pragma unroll
  for (int t = 0; t < 16; ++t)
    xv[t] = pack_f16x2_scaled(bf16_bits_to_f32(xv[t] & 0xFFFFu), bf16_bits_to_f32(xv[t] >> 16),
                              two_s);

  for (int t = 0; t < stages; ++t) {
    const int s = t % slots;
    const bool ok = mbar_wait_bounded(smem_u32(&full[s]), uint32_t((t / slots) & 1));
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) flag_error(err, kErrTimeout);
      return;
    }
    if (rslot < cnt(t)) {
      float ag = 0.f, au = 0.f;
      if (active) {
        const uint8_t* rec = ring + (size_t)s * stage_bytes + (size_t)rslot * L.bytes;
        const uint4 cg = *reinterpret_cast<const uint4*>(rec + L.gate_codes() + b * 16);
        const uint4 cu = *reinterpret_cast<const uint4*>(rec + L.up_codes() + b * 16);
        ag = dot32(cg, xv) * e8m0_to_f32(rec[L.gate_scales() + b]);
        au = dot32(cu, xv) * e8m0_to_f32(rec[L.up_scales() + b]);
      }
      const float v = warp_sum2(ag, au, lane);  // lanes 0-15: g, 16-31: u
      if ((lane & 15) == 0)
        part[((size_t)s * R + rslot) * NB * 2 + chunk * 2 + (lane >> 4)] = v * inv;
    }
    mbar_arrive(smem_u32(&empty[s]));
  }
}

// ---------------------------------------------------------------------------
// m = 1..8 (MT = 1, 2, 4 or 8 rows of x), x staged in shared memory as f16.
// x layout in shared memory: 16-byte chunk q (0..3) of block b of row i at
// ((i*4 + q) * nblk + b) * 16, so lanes reading consecutive blocks hit
// consecutive 16-byte words (no bank conflicts).
// ---------------------------------------------------------------------------
template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
    swiglu_mxfp4_mt_kernel(const uint8_t* __restrict__ packed, int n, int k, int m,
                           const uint16_t* __restrict__ x, uint16_t* __restrict__ h, int slots,
                           int32_t* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SwigluRecord L(k);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r0 = int((int64_t)n * blockIdx.x / gridDim.x);
  const int r1 = int((int64_t)n * (blockIdx.x + 1) / gridDim.x);
  const int cnt = r1 - r0;
  const int nrec = cnt > warp ? (cnt - warp + kWarps - 1) / kWarps : 0;
  const size_t ring_bytes = (size_t)kWarps * slots * L.bytes;
  uint4* xs = reinterpret_cast<uint4*>(smem + ring_bytes);            // MT * 4 * nblk chunks
  int* sxs = reinterpret_cast<int*>(smem + ring_bytes + (size_t)MT * 2 * k);  // MT exponents
  float* red = reinterpret_cast<float*>(sxs + MT);                      // MT * kWarps maxima
  uint64_t* bars_all = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(red + MT * kWarps) + 7) & ~uintptr_t(7));

  WarpRing ring;
  ring.slots = slots;
  ring.rec_bytes = L.bytes;
  ring.slot_bytes = L.bytes;
  ring.base = smem + (size_t)warp * slots * L.bytes;
  ring.bars = bars_all + warp * slots;
  ring.packed = packed;
  ring.policy = l2_evict_first_policy();
  ring.init(lane);

  pdl_allow_next_grid();
  if (lane == 0)
    for (int j = 0; j < min(slots, nrec); ++j) ring.issue_to(j, r0 + warp + j * kWarps, 1);
  pdl_wait_prior_grid();

  // Per-row max |x| -> prescale exponent; then convert x into shared memory.
  for (int i = 0; i < MT; ++i) {
    float mx = 0.f;
    if (i < m)
      for (int t = threadIdx.x; t < k; t += kThreads)
        mx = fmaxf(mx, fabsf(bf16_bits_to_f32(x[(size_t)i * k + t])));
    mx = warp_max(mx);
    if (lane == 0) red[i * kWarps + warp] = mx;
  }
  __syncthreads();
  if (threadIdx.x < MT) {
    float mx = 0.f;
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, red[threadIdx.x * kWarps + w]);
    sxs[threadIdx.x] = min(f16_prescale_exponent(mx), 127);
  }
  __syncthreads();
  const int nblk = L.nblk;
  for (int c = threadIdx.x; c < MT * 4 * nblk; c += kThreads) {
    const int i = c / (4 * nblk);
    const int rem = c - i * 4 * nblk;
    const int q = rem / nblk, b = rem - q * nblk;
    uint4 o = make_uint4(0, 0, 0, 0);
    if (i < m) {
      const float two_s = scalbnf(1.0f, sxs[i]);
      const uint4 v = *reinterpret_cast<const uint4*>(x + (size_t)i * k + b * 32 + q * 8);
      o.x = pack_f16x2_scaled(bf16_bits_to_f32(v.x & 0xFFFFu), bf16_bits_to_f32(v.x >> 16), two_s);
      o.y = pack_f16x2_scaled(bf16_bits_to_f32(v.y & 0xFFFFu), bf16_bits_to_f32(v.y >> 16), two_s);
      o.z = pack_f16x2_scaled(bf16_bits_to_f32(v.z & 0xFFFFu), bf16_bits_to_f32(v.z >> 16), two_s);
      o.w = pack_f16x2_scaled(bf16_bits_to_f32(v.w & 0xFFFFu), bf16_bits_to_f32(v.w >> 16), two_s);
    }
    xs[c] = o;
  }
  __syncthreads();

  const int nchunk = (nblk + 31) / 32;
  for (int j = 0; j < nrec; ++j) {
    const uint8_t* rec = ring.wait_next();
    if (rec == nullptr) {
      if (lane == 0) flag_error(err, kErrTimeout);
      ring.drain(j, nrec);
      return;
    }
    float ag[MT], au[MT];
#pragma unroll
    for (int i = 0; i < MT; ++i) ag[i] = au[i] = 0.f;
    for (int c = 0; c < nchunk; ++c) {
      const int b = 32 * c + lane;
      if (b < nblk) {
        uint32_t hg[16], hu[16];
        decode32(*reinterpret_cast<const uint4*>(rec + L.gate_codes() + b * 16), hg);
        decode32(*reinterpret_cast<const uint4*>(rec + L.up_codes() + b * 16), hu);
        const float sg = e8m0_to_f32(rec[L.gate_scales() + b]);
        const float su = e8m0_to_f32(rec[L.up_scales() + b]);
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          uint32_t xv[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 t = xs[(i * 4 + q) * nblk + b];
            xv[4 * q + 0] = t.x;
            xv[4 * q + 1] = t.y;
            xv[4 * q + 2] = t.z;
            xv[4 * q + 3] = t.w;
          }
          ag[i] = fmaf(dot32_decoded(hg, xv), sg, ag[i]);
          au[i] = fmaf(dot32_decoded(hu, xv), su, au[i]);
        }
      }
    }
    const float pg = *reinterpret_cast<const float*>(rec + L.post);
    const float pu = *reinterpret_cast<const float*>(rec + L.post + 4);
    __syncwarp();
    if (lane == 0 && j + slots < nrec) ring.issue_to(ring.cur, r0 + warp + (j + slots) * kWarps, 1);
    ring.advance();
    const int r = r0 + warp + j * kWarps;
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      const float v = warp_sum2(ag[i], au[i], lane);
      const float vu = __shfl_sync(0xffffffffu, v, 16);
      if (lane == 0 && i < m) {
        const float g = scalbnf(v, -sxs[i]) * pg;
        const float u = scalbnf(vu, -sxs[i]) * pu;
        h[(size_t)i * n + r] = f32_to_bf16_rne(silu_mul(g, u));
      }
    }
  }
}

template <typename Kern>
cudaError_t launch_pdl(Kern kern, int grid, int smem, cudaStream_t s, bool pdl,
                       const uint8_t* packed, int n, int k, const uint16_t* x, uint16_t* h,
                       int slots, int32_t* err) {
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
  return cudaLaunchKernelEx(&cfg, kern, packed, n, k, x, h, slots, err);
}

template <typename Kern>
cudaError_t launch_pdl_m(Kern kern, int grid, int smem, cudaStream_t s, bool pdl,
                         const uint8_t* packed, int n, int k, int m, const uint16_t* x,
                         uint16_t* h, int slots, int32_t* err) {
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
  return cudaLaunchKernelEx(&cfg, kern, packed, n, k, m, x, h, slots, err);
}

// Shared memory given to one CTA's ring: small enough that two CTAs fit on
// an SM, so the next kernel's CTA can start streaming while this one ends.
constexpr int kRingBudget = 100 * 1024;

template <int NB, int RPC>
cudaError_t run_m1(const DeviceInfo& di, const uint8_t* packed, int n, int k, const uint16_t* x,
                   uint16_t* h, cudaStream_t s, bool pdl) {
  // Two CTAs per SM (16 resident warps) with two slots per warp while x fits
  // in 128 registers; one CTA per SM with deeper rings for wider K.
  const SwigluRecord L(k);
  const int ctas_per_sm = NB <= 3 ? TT_M1_CTAS_PER_SM : 1;
  const int slot_bytes = RPC * L.bytes;
  int slots = kRingBudget / (kWarps * (slot_bytes + 8));
  slots = slots < 2 ? 2 : (slots > 4 ? 4 : slots);
  if (NB <= 3) slots = TT_M1_SLOTS;
  const int smem = kWarps * slots * (slot_bytes + 8) + 2 * k;  // ring, barriers, x
  if (smem > di.smem_optin) return cudaErrorInvalidConfiguration;
  auto kern = swiglu_mxfp4_m1_kernel<NB, RPC>;
  cudaError_t e = ensure_smem(di, kern, smem);
  if (e != cudaSuccess) return e;
  int grid = ctas_per_sm * di.sms;
  const int units = (n + RPC - 1) / RPC;
  if (grid > units) grid = units;
  return launch_pdl(kern, grid, smem, s, pdl, packed, n, k, x, h, slots, di.error_word);
}

template <typename Kern>
cudaError_t launch_threads(Kern kern, int grid, int threads, int smem, cudaStream_t s, bool pdl,
                           const uint8_t* packed, int n, int k, const uint16_t* x, uint16_t* h,
                           int slots, int32_t* err) {
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
  return cudaLaunchKernelEx(&cfg, kern, packed, n, k, x, h, slots, err);
}

// Shared memory of one CTA of the x-in-shared-memory kernel: at most half an
// SM, so that the next kernel's CTA fits beside it.
// Shared memory of one m = 1 CTA: half an SM, so that the next kernel's CTA
// (programmatic dependent launch) fits beside it.
#ifndef TT_M1_SMEM_BUDGET
#define TT_M1_SMEM_BUDGET (110 * 1024)
#endif
constexpr int kHalfSmBudget = TT_M1_SMEM_BUDGET;

template <int NB, int RPC, int WARPS>
cudaError_t run_m1x(const DeviceInfo& di, const uint8_t* packed, int n, int k, const uint16_t* x,
                    uint16_t* h, cudaStream_t s, bool pdl) {
  const SwigluRecord L(k);
  const int slot_bytes = RPC * L.bytes;
  const int fixed = 4 * k + WARPS * 4 + 16;  // raw + f16 x, per-warp maxima
  int slots = (kHalfSmBudget - fixed) / (WARPS * (slot_bytes + 8));
  if (slots > TT_M1_SLOTS) slots = TT_M1_SLOTS;
  if (slots < 1) slots = 1;
  const int smem = WARPS * slots * (slot_bytes + 8) + fixed;
  if (smem > di.smem_optin) return cudaErrorInvalidConfiguration;
  auto kern = swiglu_mxfp4_m1x_kernel<NB, RPC, WARPS>;
  cudaError_t e = ensure_smem(di, kern, smem);
  if (e != cudaSuccess) return e;
  int grid = TT_M1X_CTAS_PER_SM * di.sms;
  const int units = (n + RPC - 1) / RPC;
  if (grid > units) grid = units;
  return launch_threads(kern, grid, WARPS * 32, smem, s, pdl, packed, n, k, x, h, slots,
                        di.error_word);
}

// Stage budget of the warp-specialised kernel: under half an SM, so that
// the next kernel's CTA fits beside it.
constexpr int kStageBudget = 100 * 1024;

template <int NB>
cudaError_t run_m1s(const DeviceInfo& di, const uint8_t* packed, int n, int k, const uint16_t* x,
                    uint16_t* h, cudaStream_t s, bool pdl) {
  constexpr int R = NB >= 16 ? 1 : 16 / NB;
  constexpr int W = NB * R;
  const SwigluRecord L(k);
  const int stage_bytes = R * L.bytes;
  const int per_slot = stage_bytes + 16 + R * NB * 8;
  int slots = kStageBudget / per_slot;
  if (slots > TT_M1S_SLOTS) slots = TT_M1S_SLOTS;
  if (slots < 2) slots = 2;
  const int smem = slots * per_slot;
  if (smem > di.smem_optin) return cudaErrorInvalidConfiguration;
  auto kern = swiglu_mxfp4_m1s_kernel<NB, R>;
  cudaError_t e = ensure_smem(di, kern, smem);
  if (e != cudaSuccess) return e;
  int grid = di.sms;
  const int units = (n + R - 1) / R;
  if (grid > units) grid = units;
  return launch_threads(kern, grid, (W + 1) * 32, smem, s, pdl, packed, n, k, x, h, slots,
                        di.error_word);
}

template <int MT>
cudaError_t run_mt(const DeviceInfo& di, const uint8_t* packed, int n, int k, int m,
                   const uint16_t* x, uint16_t* h, cudaStream_t s, bool pdl) {
  const SwigluRecord L(k);
  const int xs_bytes = MT * 2 * k + MT * 4 + MT * kWarps * 4 + 16;
  const int avail = di.smem_optin - xs_bytes;
  const int per_slot = kWarps * (L.bytes + 8);
  int slots = (avail < kRingBudget ? avail : kRingBudget) / per_slot;
  if (slots < 2) slots = avail / per_slot < 2 ? avail / per_slot : 2;  // wide K: use more smem
  if (slots < 1) return cudaErrorInvalidConfiguration;
  if (slots > 6) slots = 6;
  const int smem = kWarps * slots * (L.bytes + 8) + xs_bytes;
  auto kern = swiglu_mxfp4_mt_kernel<MT>;
  cudaError_t e = ensure_smem(di, kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = n < di.sms ? n : di.sms;
  return launch_pdl_m(kern, grid, smem, s, pdl, packed, n, k, m, x, h, slots, di.error_word);
}

}  // namespace

cudaError_t launch_swiglu_mxfp4_cc(const uint8_t* packed, int n, int k, const uint16_t* x, int m,
                                   uint16_t* h, cudaStream_t s, bool pdl) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorNoDevice;
  if (m == 1 && TT_M1_STAGED) {
    switch ((k / 32 + 31) / 32) {
      case 1: return run_m1s<1>(*di, packed, n, k, x, h, s, pdl);
      case 2: return run_m1s<2>(*di, packed, n, k, x, h, s, pdl);
      case 3: return run_m1s<3>(*di, packed, n, k, x, h, s, pdl);
      case 4: return run_m1s<4>(*di, packed, n, k, x, h, s, pdl);
      case 5: return run_m1s<5>(*di, packed, n, k, x, h, s, pdl);
      case 6: return run_m1s<6>(*di, packed, n, k, x, h, s, pdl);
      case 7: return run_m1s<7>(*di, packed, n, k, x, h, s, pdl);
      case 8: return run_m1s<8>(*di, packed, n, k, x, h, s, pdl);
      case 9: return run_m1s<9>(*di, packed, n, k, x, h, s, pdl);
      case 10: return run_m1s<10>(*di, packed, n, k, x, h, s, pdl);
      case 11: return run_m1s<11>(*di, packed, n, k, x, h, s, pdl);
      case 12: return run_m1s<12>(*di, packed, n, k, x, h, s, pdl);
      case 13: return run_m1s<13>(*di, packed, n, k, x, h, s, pdl);
      case 14: return run_m1s<14>(*di, packed, n, k, x, h, s, pdl);
      case 15: return run_m1s<15>(*di, packed, n, k, x, h, s, pdl);
      case 16: return run_m1s<16>(*di, packed, n, k, x, h, s, pdl);
      default: break;
    }
  }
  if (m == 1 && TT_M1_XSMEM) {
    const int nb = (k / 32 + 31) / 32;
    switch (nb) {
      case 1: return run_m1x<1, TT_M1_RPC, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 2: return run_m1x<2, TT_M1_RPC, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 3: return run_m1x<3, TT_M1_RPC, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 4: return run_m1x<4, 1, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 5: return run_m1x<5, 1, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 6: return run_m1x<6, 1, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 7: return run_m1x<7, 1, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 8: return run_m1x<8, 1, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      default: break;
    }
  }
  if (m == 1) {
    const int nb = (k / 32 + 31) / 32;
    switch (nb) {
      case 1: return run_m1<1, TT_M1_RPC>(*di, packed, n, k, x, h, s, pdl);
      case 2: return run_m1<2, TT_M1_RPC>(*di, packed, n, k, x, h, s, pdl);
      case 3: return run_m1<3, TT_M1_RPC>(*di, packed, n, k, x, h, s, pdl);
      case 4: return run_m1<4, 1>(*di, packed, n, k, x, h, s, pdl);
      case 5: return run_m1<5, 1>(*di, packed, n, k, x, h, s, pdl);
      case 6: return run_m1<6, 1>(*di, packed, n, k, x, h, s, pdl);
      default: return run_mt<1>(*di, packed, n, k, 1, x, h, s, pdl);
    }
  }
  if (m == 2) return run_mt<2>(*di, packed, n, k, m, x, h, s, pdl);
  if (m <= 4) return run_mt<4>(*di, packed, n, k, m, x, h, s, pdl);
  if (m <= 8) return run_mt<8>(*di, packed, n, k, m, x, h, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace tt
