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
//    prescale, per 32-block at m = 1, per batch row at m = 2..8) and reused
//    for every row;
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

// Launch shape of the m = 1 kernel: ring slots per warp, records per bulk
// copy and warps per CTA (2, 1, 16 measured best; deeper rings, 2 records per
// copy, 12 or 20 warps were slower).
#ifndef TT_M1_SLOTS
#define TT_M1_SLOTS 2
#endif
#ifndef TT_M1_RPC
#define TT_M1_RPC 1
#endif
#ifndef TT_M1_WARPS
#define TT_M1_WARPS 16
#endif
// When the m = 1 kernel allows the dependent launch: 0 = at entry (measured
// best), 1 = once x has been staged.
#ifndef TT_M1_LATE_TRIGGER
#define TT_M1_LATE_TRIGGER 0
#endif
// Each CTA prefetches its whole weight range into L2 at launch (measured: no
// gain; the records phase is issue-bound).
#ifndef TT_M1_L2PF
#define TT_M1_L2PF 0
#endif

// ---------------------------------------------------------------------------
// m = 1, x staged once per CTA in shared memory as f16 (each 32-block
// prescaled by its own power of two), laid out chunk-major: 16-byte chunk q
// (0..3) of block b at xs[q*nblk + b], so a warp reading blocks b..b+31
// touches 32 consecutive 16-byte words.
// Keeping x out of registers lets WARPS warps per CTA stay resident while
// the next kernel's CTA (programmatic dependent launch) shares the SM.
// NB = number of 1024-wide K chunks; RPC = records per bulk copy; KC = K
// when it is fixed at compile time (0: K is the runtime argument), which
// turns every record and x offset into an immediate; FULL = K is exactly
// 1024 * NB, so every lane owns a block in every chunk and the per-block
// bounds tests drop out (measured: 6.46 against 6.77 us on the SmolLM3
// gate/up layer, the difference being integer and branch instructions).
// ---------------------------------------------------------------------------
template <int NB, int RPC, int WARPS, int KC, bool FULL>
__global__ void __launch_bounds__(WARPS * 32, 2)
    swiglu_mxfp4_m1x_kernel(const uint8_t* __restrict__ packed, int n, int k_arg,
                            const uint16_t* __restrict__ x, uint16_t* __restrict__ h, int slots,
                            int32_t* err) {
  static_assert(KC == 0 || (KC % 32 == 0 && (KC + 1023) / 1024 == NB), "KC and NB disagree");
  static_assert(!FULL || KC == 0 || KC == 1024 * NB, "FULL needs K == 1024 * NB");
  constexpr int THREADS = WARPS * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const int k = KC > 0 ? KC : k_arg;
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
  uint4* xs = reinterpret_cast<uint4*>(smem + ring_bytes + (size_t)WARPS * slots * 8);
  float* xinv = reinterpret_cast<float*>(xs + (k >> 3));  // [nblk] 2^-s of each x block
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

  // x: one global read per CTA.  Each 32-block of x gets its own exact
  // power-of-two prescale 2^s (its max |x| -> [2^14, 2^15)) and is stored as
  // f16 in the chunk-major layout; four threads share a block (one 16-byte
  // chunk each) and meet in two shuffles.  2^-s is folded into the block's
  // E8M0 scale below.
  const int nchunk16 = k >> 3;
  const uint64_t x_policy = l2_evict_last_policy();
  for (int c0 = 0; c0 < nchunk16; c0 += THREADS) {  // uniform trip count
    const int c = c0 + threadIdx.x;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (c < nchunk16) v = ld_global_v4_hint(reinterpret_cast<const uint4*>(x) + c, x_policy);
    float mx = fmaxf(fmaxf(fmaxf(fabsf(bf16_bits_to_f32(v.x & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.x >> 16))),
                           fmaxf(fabsf(bf16_bits_to_f32(v.y & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.y >> 16)))),
                     fmaxf(fmaxf(fabsf(bf16_bits_to_f32(v.z & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.z >> 16))),
                           fmaxf(fabsf(bf16_bits_to_f32(v.w & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.w >> 16)))));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (c < nchunk16) {
      const int sb = min(f16_prescale_exponent(mx), 127);
      const float two_s = scalbnf(1.0f, sb);
      uint4 o;
      o.x = pack_f16x2_scaled(bf16_bits_to_f32(v.x & 0xFFFFu), bf16_bits_to_f32(v.x >> 16), two_s);
      o.y = pack_f16x2_scaled(bf16_bits_to_f32(v.y & 0xFFFFu), bf16_bits_to_f32(v.y >> 16), two_s);
      o.z = pack_f16x2_scaled(bf16_bits_to_f32(v.z & 0xFFFFu), bf16_bits_to_f32(v.z >> 16), two_s);
      o.w = pack_f16x2_scaled(bf16_bits_to_f32(v.w & 0xFFFFu), bf16_bits_to_f32(v.w >> 16), two_s);
      xs[(c & 3) * L.nblk + (c >> 2)] = o;  // chunk q = c % 4 of block b = c / 4
      if ((c & 3) == 0) xinv[c >> 2] = scalbnf(1.0f, -sb);  // exact power of two
    }
  }
  __syncthreads();
  if (TT_M1_LATE_TRIGGER) pdl_allow_next_grid();
  float xi[NB];  // this lane's blocks' 2^-s
#pragma unroll
  for (int i = 0; i < NB; ++i) xi[i] = (FULL || 32 * i + lane < L.nblk) ? xinv[32 * i + lane] : 0.f;
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
      if (FULL || b < L.nblk) {
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
          if (RPC == 1 || rr < count) {  // a one-record item always holds its record
            const uint8_t* rec = slot + rr * L.bytes;
            const uint4 cg = *reinterpret_cast<const uint4*>(rec + L.gate_codes() + b * 16);
            const uint4 cu = *reinterpret_cast<const uint4*>(rec + L.up_codes() + b * 16);
            const float sg = e8m0_to_f32(rec[L.gate_scales() + b]) * xi[i];  // exact
            const float su = e8m0_to_f32(rec[L.up_scales() + b]) * xi[i];
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
      ep.put(v, 0, 8, pg[0], pu[0], 1.0f, first, lane);
      if (count > 1) ep.put(v, 16, 24, pg[1], pu[1], 1.0f, first + 1, lane);
    } else {
      const float v = warp_sum2(ag[0], au[0], lane);  // lanes 0-15: g, 16-31: u
      if (ep.fill > 31) ep.flush(h);
      ep.put(v, 0, 16, pg[0], pu[0], 1.0f, first, lane);
    }
  }
  ep.flush(h);
}

// ---------------------------------------------------------------------------
// m = 1 with K fixed at compile time, records in registers (SmolLM3-3B's
// gate/up, K = 2048: three CTAs of 8 warps per SM, 80 registers a thread;
// Phi-4's, K = 5120: two, 96 registers), warp w of the grid takes
// records w, w + (warps of the grid), ...; each lane keeps the one record it
// is about to compute in registers (its two 16-byte code chunks of each
// matrix, their scale bytes and the postscales, all requested with plain
// loads, evict-first), and requests the warp's next record as soon as the
// current one is in the multiply-adds.  The first record of every warp is
// requested before the dependency wait.  x is staged once per CTA as in
// the ring kernel above, and the arithmetic and reductions are the same, so
// the results are bit-identical to it.  No barriers, copies or waits on the
// record path: the 24 warps per SM hide each record's latency.  Measured on
// the SmolLM3 layer (rotating copies): 5.67 us, against 6.46 for the ring
// kernel; 4 CTAs per SM (64 registers) 6.15, 3 CTAs with 2 records in
// flight 6.30, 2 CTAs 6.30 to 6.46, 1 CTA 8.35 to 8.82, and 3 CTAs with a
// fourth slot left free for the next kernel's CTA 6.93.  Phi-4's layer
// (K = 5120, N = 17920): 19.8 us against 21.2 for the ring kernel.
// ---------------------------------------------------------------------------
constexpr int kRegWarps = 8;

template <int NB>
struct RegRecord {
  uint4 cg[NB], cu[NB];     // this lane's gate / up code chunks
  uint32_t sg[NB], su[NB];  // their E8M0 bytes
  float2 post;              // (post_g, post_u), the same for every lane
};

template <int KC, int CTAS>  // CTAS: CTAs per SM (the register budget of a record)
__global__ void __launch_bounds__(kRegWarps * 32, CTAS)
    swiglu_mxfp4_m1r_kernel(const uint8_t* __restrict__ packed, int n,
                            const uint16_t* __restrict__ x, uint16_t* __restrict__ h) {
  constexpr int THREADS = kRegWarps * 32;
  static_assert(KC % 1024 == 0, "whole warps in the x staging loop");
  constexpr int NB = KC / 1024;
  __shared__ __align__(16) uint4 xs[KC / 8];  // f16 x, chunk-major (as the ring kernel)
  __shared__ float xinv[KC / 32];             // 2^-s of each x block
  const SwigluRecord L(KC);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gw = blockIdx.x * kRegWarps + warp, nw = gridDim.x * kRegWarps;
  const int nitems = n > gw ? (n - gw + nw - 1) / nw : 0;
  const uint64_t pol = l2_evict_first_policy();
  auto load = [&](RegRecord<NB>& R, int rec_idx) {
    const uint8_t* rec = packed + (size_t)rec_idx * L.bytes;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int b = 32 * i + lane;
      R.cg[i] = ld_global_v4_hint(rec + L.gate_codes() + 16 * b, pol);
      R.cu[i] = ld_global_v4_hint(rec + L.up_codes() + 16 * b, pol);
      R.sg[i] = __ldcs(rec + L.gate_scales() + b);
      R.su[i] = __ldcs(rec + L.up_scales() + b);
    }
    R.post = __ldcs(reinterpret_cast<const float2*>(rec + L.post));
  };
  pdl_allow_next_grid();
  RegRecord<NB> R;
  if (nitems > 0) load(R, gw);  // weights do not depend on the previous kernel
  pdl_wait_prior_grid();

  // x: one coherent read per CTA, each 32-block prescaled by its own 2^s
  for (int c = threadIdx.x; c < KC / 8; c += THREADS) {  // 16-byte chunk c = 4 b + q of x
    const uint4 v = ld_global_v4_hint(reinterpret_cast<const uint4*>(x) + c, l2_evict_last_policy());
    float mx = fmaxf(fmaxf(fmaxf(fabsf(bf16_bits_to_f32(v.x & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.x >> 16))),
                           fmaxf(fabsf(bf16_bits_to_f32(v.y & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.y >> 16)))),
                     fmaxf(fmaxf(fabsf(bf16_bits_to_f32(v.z & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.z >> 16))),
                           fmaxf(fabsf(bf16_bits_to_f32(v.w & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.w >> 16)))));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const int sb = min(f16_prescale_exponent(mx), 127);
    const float two_s = scalbnf(1.0f, sb);
    uint4 o;
    o.x = pack_f16x2_scaled(bf16_bits_to_f32(v.x & 0xFFFFu), bf16_bits_to_f32(v.x >> 16), two_s);
    o.y = pack_f16x2_scaled(bf16_bits_to_f32(v.y & 0xFFFFu), bf16_bits_to_f32(v.y >> 16), two_s);
    o.z = pack_f16x2_scaled(bf16_bits_to_f32(v.z & 0xFFFFu), bf16_bits_to_f32(v.z >> 16), two_s);
    o.w = pack_f16x2_scaled(bf16_bits_to_f32(v.w & 0xFFFFu), bf16_bits_to_f32(v.w >> 16), two_s);
    xs[(c & 3) * L.nblk + (c >> 2)] = o;  // chunk q = c % 4 of block b = c / 4
    if ((c & 3) == 0) xinv[c >> 2] = scalbnf(1.0f, -sb);  // exact power of two
  }
  __syncthreads();
  float xi[NB];  // this lane's blocks' 2^-s
#pragma unroll
  for (int i = 0; i < NB; ++i) xi[i] = xinv[32 * i + lane];

  for (int j = 0; j < nitems; ++j) {
    float ag = 0.f, au = 0.f;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int b = 32 * i + lane;
      uint32_t xv[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 t = xs[q * L.nblk + b];
        xv[4 * q + 0] = t.x;
        xv[4 * q + 1] = t.y;
        xv[4 * q + 2] = t.z;
        xv[4 * q + 3] = t.w;
      }
      ag = fmaf(dot32(R.cg[i], xv), e8m0_to_f32(R.sg[i]) * xi[i], ag);  // exact factor
      au = fmaf(dot32(R.cu[i], xv), e8m0_to_f32(R.su[i]) * xi[i], au);
    }
    const float pg = R.post.x, pu = R.post.y;
    const int rec = gw + j * nw;
    if (j + 1 < nitems) load(R, rec + nw);  // the warp's next record
    const float v = warp_sum2(ag, au, lane);  // lanes 0-15: g, 16-31: u
    const float g = __shfl_sync(0xffffffffu, v, 0) * pg;
    const float u = __shfl_sync(0xffffffffu, v, 16) * pu;
    if (lane == 0) h[rec] = f32_to_bf16_rne(silu_mul(g, u));
  }
}

template <int KC, int CTAS>
cudaError_t run_m1r(const DeviceInfo& di, const uint8_t* packed, int n, const uint16_t* x,
                    uint16_t* h, cudaStream_t s, bool pdl) {
  int grid = CTAS * di.sms;
  const int need = (n + kRegWarps - 1) / kRegWarps;
  if (grid > need) grid = need;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRegWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, swiglu_mxfp4_m1r_kernel<KC, CTAS>, packed, n, x, h);
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
        mx = fmaxf(mx, fabsf(bf16_bits_to_f32(__ldca(x + (size_t)i * k + t))));
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
      const uint4 v = __ldca(reinterpret_cast<const uint4*>(x + (size_t)i * k + b * 32 + q * 8));
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

// Shared memory of one m = 1 CTA: half an SM, so that the next kernel's CTA
// (programmatic dependent launch) fits beside it.
#ifndef TT_M1_SMEM_BUDGET
#define TT_M1_SMEM_BUDGET (110 * 1024)
#endif
constexpr int kHalfSmBudget = TT_M1_SMEM_BUDGET;

template <int NB, int RPC, int WARPS, int KC = 0, bool FULL = false>
cudaError_t run_m1x(const DeviceInfo& di, const uint8_t* packed, int n, int k, const uint16_t* x,
                    uint16_t* h, cudaStream_t s, bool pdl) {
  const SwigluRecord L(k);
  const int slot_bytes = RPC * L.bytes;
  const int fixed = 2 * k + 4 * L.nblk + 16;  // f16 x, per-block factors
  int slots = (kHalfSmBudget - fixed) / (WARPS * (slot_bytes + 8));
  if (slots > TT_M1_SLOTS) slots = TT_M1_SLOTS;
  if (slots < 1) slots = 1;
  const int smem = WARPS * slots * (slot_bytes + 8) + fixed;
  if (smem > di.smem_optin) return cudaErrorInvalidConfiguration;
  auto kern = swiglu_mxfp4_m1x_kernel<NB, RPC, WARPS, KC, FULL>;
  cudaError_t e = ensure_smem(di, kern, smem);
  if (e != cudaSuccess) return e;
  int grid = di.sms;  // one CTA per SM
  const int units = (n + RPC - 1) / RPC;
  if (grid > units) grid = units;
  return launch_threads(kern, grid, WARPS * 32, smem, s, pdl, packed, n, k, x, h, slots,
                        di.error_word);
}

// Shared memory given to one CTA's ring of the m = 2..8 kernel: small enough
// that two CTAs fit on an SM, so the next kernel's CTA can start streaming
// while this one ends.
constexpr int kRingBudget = 100 * 1024;

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
  if (m == 1) {
    // K of the gate/up layers of the models the library serves get the
    // register kernel with K fixed (SmolLM3-3B's 2048 at three CTAs per SM,
    // Phi-4's 5120, whose records take more registers, at two); every other K
    // takes the runtime-K ring kernel, without per-block bounds tests when
    // K % 1024 == 0.
    if (k == 2048) return run_m1r<2048, 3>(*di, packed, n, x, h, s, pdl);
    if (k == 5120) return run_m1r<5120, 2>(*di, packed, n, x, h, s, pdl);
    if (k % 1024 == 0) {
      switch (k / 1024) {
        case 1: return run_m1x<1, TT_M1_RPC, TT_M1_WARPS, 0, true>(*di, packed, n, k, x, h, s, pdl);
        case 3: return run_m1x<3, TT_M1_RPC, TT_M1_WARPS, 0, true>(*di, packed, n, k, x, h, s, pdl);
        case 4: return run_m1x<4, 1, TT_M1_WARPS, 0, true>(*di, packed, n, k, x, h, s, pdl);
        case 8: return run_m1x<8, 1, TT_M1_WARPS, 0, true>(*di, packed, n, k, x, h, s, pdl);
        default: break;  // 6 and 7 chunks: the runtime kernel below
      }
    }
    switch ((k / 32 + 31) / 32) {
      case 1: return run_m1x<1, TT_M1_RPC, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 2: return run_m1x<2, TT_M1_RPC, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 3: return run_m1x<3, TT_M1_RPC, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 4: return run_m1x<4, 1, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 5: return run_m1x<5, 1, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 6: return run_m1x<6, 1, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 7: return run_m1x<7, 1, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      case 8: return run_m1x<8, 1, TT_M1_WARPS>(*di, packed, n, k, x, h, s, pdl);
      default: return run_mt<1>(*di, packed, n, k, 1, x, h, s, pdl);  // k > 8192
    }
  }
  if (m == 2) return run_mt<2>(*di, packed, n, k, m, x, h, s, pdl);
  if (m <= 4) return run_mt<4>(*di, packed, n, k, m, x, h, s, pdl);
  if (m <= 8) return run_mt<8>(*di, packed, n, k, m, x, h, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace tt
