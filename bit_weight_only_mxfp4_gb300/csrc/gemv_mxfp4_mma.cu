// MXFP4 gate/up SwiGLU matvec for small batches (m = 2..8), with the
// multiply-adds on the warp-level tensor-core instruction (mma.sync m16n8k16,
// f16 x f16 -> fp32).
//
// Method: ThinTensor devlog (kerbin.cskartikey.dev/@satvikhardat), Dev Log #4
// "Where Blackwell helps": read the MXFP4 bytes, use the block scales,
// multiply against bf16 activations, accumulate safely, then apply the row
// postscale; the gate/up pair feeds the gated activation of Dev Log #2.
// Decode is a weight-read problem (Dev Log #4, "Why gate/up was the right
// target"): the kernel must stream the packed bytes once at HBM speed.  With
// m > 1 rows of x, one decoded weight feeds m multiply-adds; on the FMA pipe
// that keeps the CUDA-core kernels ALU-bound from m = 2 on.  Here the
// multiply-adds go to the tensor pipe instead: a warp decodes its E2M1 codes
// with cvt.rn.f16x2.e2m1x2 straight into MMA A fragments, and one mma.sync
// serves all m rows of x (the MMA's 8 columns), so the issue cost per weight
// no longer grows with m.  The work stays a stream bound by HBM.
//
//  * persistent grid, one CTA per SM, each CTA owning a contiguous range of
//    output rows, taken in tiles of 8 rows (8 packed records, layout.cuh);
//  * a copy warp runs a ring of S tile slots in shared memory, filled by bulk
//    copies (TMA, non-tensor) signalled on an mbarrier; the first tiles are
//    requested before the programmatic-dependent-launch wait, so weight
//    streaming overlaps the previous kernel's tail;
//  * 16 consumer warps split K: warp w owns the 32-blocks w, w+16, w+32, ...,
//    so its slice of x is converted once into MMA B fragments held in
//    registers for the whole kernel (f16 after an exact power-of-two prescale
//    per 32-block and batch row, the block max |x| -> [2^14, 2^15));
//  * A fragments: rows 0..7 are the gate rows of the tile's 8 output rows,
//    rows 8..15 the matching up rows; B column c is batch row c.  Within a
//    32-block the reduction order is free, so the two MMAs of a block take
//    the 4 code bytes 4t..4t+3 of each row (k = 8t .. 8t+7) with one 32-bit
//    load per row, and x is staged in the same order;
//  * each 32-block's D is scaled once in fp32 by its E8M0 factor times the x
//    block's 2^-s (both exact powers of two); the warps' partial sums meet in
//    shared memory, and an epilogue warp adds them in a fixed order, applies
//    the postscales and SwiGLU, and stores bf16.
//
// e2m1 x f16 products are exact; the tensor core accumulates in fp32.
#include "common.cuh"
#include "launch.h"
#include "layout.cuh"
#include "mxfp4_core.cuh"

namespace tt {
namespace {

// Consumer warps (the K split) and the 32-blocks each holds in registers
// (K <= 5120); then one copy warp and one epilogue warp.
constexpr int kMmaWarps = 16;
constexpr int kCopyWarp = kMmaWarps, kEpiWarp = kMmaWarps + 1;
constexpr int kMmaThreads = (kMmaWarps + 2) * 32;
constexpr int kMmaMaxNbw = 10;
constexpr int kTileRows = 8;
// Shared memory of one CTA: half an SM, so that the next kernel's CTA
// (programmatic dependent launch) fits beside it.
#ifndef TT_MMA_SMEM_BUDGET
#define TT_MMA_SMEM_BUDGET (110 * 1024)
#endif
#ifndef TT_MMA_MAX_SLOTS
#define TT_MMA_MAX_SLOTS 6
#endif

// Shared-memory loads as plain C++ accesses: the compiler schedules them
// freely among the decode and MMA work, but never across the mbarrier waits
// (asm with a memory clobber) that make the slot's bytes visible.
__device__ __forceinline__ uint32_t lds_u32(const uint8_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}
__device__ __forceinline__ uint32_t lds_u8(const uint8_t* p) { return *p; }

__device__ __forceinline__ float bf16_abs_max8(const uint4& v) {
  return fmaxf(fmaxf(fmaxf(fabsf(bf16_bits_to_f32(v.x & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.x >> 16))),
                     fmaxf(fabsf(bf16_bits_to_f32(v.y & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.y >> 16)))),
               fmaxf(fmaxf(fabsf(bf16_bits_to_f32(v.z & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.z >> 16))),
                     fmaxf(fabsf(bf16_bits_to_f32(v.w & 0xFFFFu)), fabsf(bf16_bits_to_f32(v.w >> 16)))));
}
// 8 bf16 -> 4 f16x2 after the exact prescale two_s
__device__ __forceinline__ void bf16x8_to_f16x2(const uint4& v, float two_s, uint32_t* o) {
  o[0] = pack_f16x2_scaled(bf16_bits_to_f32(v.x & 0xFFFFu), bf16_bits_to_f32(v.x >> 16), two_s);
  o[1] = pack_f16x2_scaled(bf16_bits_to_f32(v.y & 0xFFFFu), bf16_bits_to_f32(v.y >> 16), two_s);
  o[2] = pack_f16x2_scaled(bf16_bits_to_f32(v.z & 0xFFFFu), bf16_bits_to_f32(v.z >> 16), two_s);
  o[3] = pack_f16x2_scaled(bf16_bits_to_f32(v.w & 0xFFFFu), bf16_bits_to_f32(v.w >> 16), two_s);
}

// Partial sums per consumer warp and slot: every lane's 4 D values.  After
// them, per slot, the tile's postscales [8 rows][gate, up], copied out by
// consumer warp 0.
constexpr int kPartialFloats = 128;

// Shared-memory plan, identical on host and device.
struct MmaPlan {
  int stride;       // bytes between two records of a tile slot (record + pad)
  int slot_bytes;   // kTileRows * stride
  int part_bytes;   // per slot
  int slots;
  int smem;
  __host__ __device__ MmaPlan(int k, int nslots) {
    const SwigluRecord L(k);
    // An odd multiple of 16 bytes between records puts the 8 rows of a tile
    // on different bank groups (conflict-free code loads).
    stride = L.bytes + ((L.bytes & 31) == 0 ? 16 : 0);
    slot_bytes = kTileRows * stride;
    part_bytes = kMmaWarps * kPartialFloats * 4 + 2 * kTileRows * 4;  // + postscales
    slots = nslots;
    smem = slots * (slot_bytes + part_bytes) + 3 * slots * 8;
  }
};

// The CTA's view of its ring and its row range.
struct Ring {
  SwigluRecord L;
  MmaPlan P;
  int S, r0, r1, ntiles, active;
  uint8_t* slots;
  float* parts;
  uint64_t *full, *empty, *reduced;  // data landed / slot read / partials summed
  __device__ Ring(uint8_t* smem, int n, int k, int nslots, int active_)
      : L(k), P(k, nslots), S(nslots), active(active_) {
    r0 = int((int64_t)n * blockIdx.x / gridDim.x);
    r1 = int((int64_t)n * (blockIdx.x + 1) / gridDim.x);
    ntiles = (r1 - r0 + kTileRows - 1) / kTileRows;
    slots = smem;
    parts = reinterpret_cast<float*>(smem + (size_t)S * P.slot_bytes);
    full = reinterpret_cast<uint64_t*>(smem + (size_t)S * (P.slot_bytes + P.part_bytes));
    empty = full + S;
    reduced = empty + S;
  }
  __device__ void init() const {
    if (threadIdx.x == 0) {
      for (int s = 0; s < S; ++s) {
        mbar_init(smem_u32(&full[s]), 1);
        mbar_init(smem_u32(&empty[s]), active);
        mbar_init(smem_u32(&reduced[s]), 1);
      }
      fence_mbar_init();
    }
    __syncthreads();
  }
};

// ---------------------------------------------------------------------------
// Copy warp: requests the first tiles before the dependency wait, then
// refills each slot as soon as every consumer has released it.
// ---------------------------------------------------------------------------
__device__ void copy_warp(const Ring& R, const uint8_t* __restrict__ packed, int32_t* err) {
  const int lane = threadIdx.x & 31;
  const uint64_t pol = l2_evict_first_policy();
  const bool contiguous = R.P.stride == R.L.bytes;
  auto issue = [&](int tile, int s) {
    const int rb = R.r0 + tile * kTileRows;
    const int cnt = min(kTileRows, R.r1 - rb);
    const uint32_t bar = smem_u32(&R.full[s]);
    const uint32_t dst = smem_u32(R.slots + (size_t)s * R.P.slot_bytes);
    const uint8_t* src = packed + (int64_t)rb * R.L.bytes;
    if (contiguous) {  // one copy of the tile's records
      if (lane == 0) {
        mbar_arrive_expect_tx(bar, uint32_t(cnt * R.L.bytes));
        bulk_g2s(dst, src, uint32_t(cnt * R.L.bytes), bar, pol);
      }
    } else {  // padded slot: lanes 0..7 copy one record each
      if (lane == 0) mbar_arrive_expect_tx(bar, uint32_t(cnt * R.L.bytes));
      __syncwarp();
      if (lane < cnt)
        bulk_g2s(dst + uint32_t(lane * R.P.stride), src + (int64_t)lane * R.L.bytes,
                 uint32_t(R.L.bytes), bar, pol);
    }
  };
  for (int j = 0; j < min(R.S, R.ntiles); ++j) issue(j, j);  // before the dependency wait
  int issued = min(R.S, R.ntiles);  // tiles requested so far
  int s = 0;
  uint32_t ph = 0;
  for (int j = 0; j + R.S < R.ntiles; ++j) {
    const bool ok = mbar_wait_bounded(smem_u32(&R.empty[s]), ph);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) flag_error(err, kErrTimeout);
      break;
    }
    __syncwarp();
    issue(j + R.S, s);
    issued = j + R.S + 1;
    if (++s == R.S) {
      s = 0;
      ph ^= 1u;
    }
  }
  // Only the last copy into each slot can still be in flight (each earlier
  // one was consumed before its slot was refilled): let those land before
  // the CTA may exit.  Normally they already have.
  for (int ss = 0; ss < R.S && ss < issued; ++ss) {
    const int last = issued - 1 - ((issued - 1 - ss) % R.S);
    (void)mbar_wait_bounded(smem_u32(&R.full[ss]), uint32_t((last / R.S) & 1));
  }
}

// ---------------------------------------------------------------------------
// Epilogue warp: for every released tile, sums the consumers' partials in a
// fixed order, applies the postscales and SwiGLU, and stores h.
// ---------------------------------------------------------------------------
__device__ void epilogue_warp(const Ring& R, int n, int m, uint16_t* __restrict__ h,
                              int32_t* err) {
  const int lane = threadIdx.x & 31;
  pdl_wait_prior_grid();  // h may still be read by the previous kernel
  const int g = lane >> 2, t = lane & 3;
  int s = 0;
  uint32_t ph = 0;
  for (int j = 0; j < R.ntiles; ++j) {
    const bool ok = mbar_wait_bounded(smem_u32(&R.empty[s]), ph);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) flag_error(err, kErrTimeout);
      return;
    }
    const int rb = R.r0 + j * kTileRows;
    const int cnt = min(kTileRows, R.r1 - rb);
    const float* pp = R.parts + (size_t)s * (R.P.part_bytes / 4);
    const float2 post = *reinterpret_cast<const float2*>(pp + kMmaWarps * kPartialFloats + 2 * g);
    // lane (g, t) holds rows g (gate, up) x batch columns 2t, 2t+1
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    for (int w = 0; w < R.active; ++w) {
      const float4 v = *reinterpret_cast<const float4*>(pp + w * kPartialFloats + lane * 4);
      a0 += v.x;
      a1 += v.y;
      a2 += v.z;
      a3 += v.w;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&R.reduced[s]));  // partials consumed
    if (g < cnt) {
      const int c0 = 2 * t, c1 = 2 * t + 1;
      if (c0 < m) h[(size_t)c0 * n + rb + g] = f32_to_bf16_rne(silu_mul(a0 * post.x, a2 * post.y));
      if (c1 < m) h[(size_t)c1 * n + rb + g] = f32_to_bf16_rne(silu_mul(a1 * post.x, a3 * post.y));
    }
    if (++s == R.S) {
      s = 0;
      ph ^= 1u;
    }
  }
}

// A consumer's hand-over of one tile: wait until the epilogue warp has summed
// the slot's previous partials (from the second round on), write this
// tile's (warp 0 also copies the tile's postscales out of the slot, which is
// refilled as soon as every consumer has released it), and release the slot.
// False after a timeout (warp-uniform).
template <class Write>
__device__ __forceinline__ bool hand_over(const Ring& R, int j, int s, uint32_t ph, int lane,
                                          int warp, Write write) {
  if (j >= R.S && !__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&R.reduced[s]), ph ^ 1u)))
    return false;
  write();
  if (warp == 0 && lane < 2 * kTileRows) {
    const float* rec = reinterpret_cast<const float*>(
        R.slots + (size_t)s * R.P.slot_bytes + (size_t)(lane >> 1) * R.P.stride + R.L.post);
    R.parts[(size_t)s * (R.P.part_bytes / 4) + (R.P.part_bytes / 4 - 2 * kTileRows) + lane] =
        rec[lane & 1];
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&R.empty[s]));  // slot read, partials written
  return true;
}

// ---------------------------------------------------------------------------
// m = 2..8: B column c = batch row c.  NBW = 32-blocks per consumer warp.
// ---------------------------------------------------------------------------
template <int NBW>
__global__ void __launch_bounds__(kMmaThreads, 1)
    swiglu_mxfp4_mma_kernel(const uint8_t* __restrict__ packed, int n, int k, int m,
                            const uint16_t* __restrict__ x, uint16_t* __restrict__ h, int nslots,
                            int32_t* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int nblk = k >> 5;
  const int active = min(kMmaWarps, nblk);  // consumer warps that own blocks
  const Ring R(smem, n, k, nslots, active);
  R.init();
  pdl_allow_next_grid();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == kCopyWarp) {
    copy_warp(R, packed, err);
    return;
  }
  if (warp == kEpiWarp) {
    epilogue_warp(R, n, m, h, err);
    return;
  }
  if (warp >= active) return;
  pdl_wait_prior_grid();
  const int g = lane >> 2, t = lane & 3;
  const int cnt = (nblk - warp + kMmaWarps - 1) / kMmaWarps;  // this warp's blocks

  // x: this warp's blocks (w, w + 16, ...) of every batch row, converted
  // once into B fragments: thread (g, t) holds x[g][32b + 8t .. 8t+7] of
  // block b; the 4 lanes of a row meet in two shuffles for the block max.
  uint32_t xb[NBW][4];
  float xs0[NBW], xs1[NBW];  // 2^-s of batch columns 2t and 2t+1 per block
#pragma unroll
  for (int j = 0; j < NBW; ++j) {
    const int b = warp + kMmaWarps * j;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (j < cnt && g < m)
      v = __ldcg(reinterpret_cast<const uint4*>(x + (size_t)g * k + 32 * b + 8 * t));
    float mx = bf16_abs_max8(v);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const int sb = min(f16_prescale_exponent(mx), 127);
    bf16x8_to_f16x2(v, scalbnf(1.0f, sb), xb[j]);
    const float inv = scalbnf(1.0f, -sb);  // exact power of two
    // batch column c's factor sits on lane 4c (row g = c, t = 0)
    xs0[j] = __shfl_sync(0xffffffffu, inv, 8 * t);
    xs1[j] = __shfl_sync(0xffffffffu, inv, 8 * t + 4);
  }

  const int row_off = g * R.P.stride + 4 * t;
  const int up_off = R.L.up_codes();
  const int gs_off = R.L.gate_scales() - 4 * t;  // scale bytes: no t term
  const int us_off = R.L.up_scales() - 4 * t;
  float* mypart = R.parts + (size_t)warp * kPartialFloats + lane * 4;

  int s = 0;
  uint32_t ph = 0;
  for (int j = 0; j < R.ntiles; ++j) {
    const bool ok = mbar_wait_bounded(smem_u32(&R.full[s]), ph);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) flag_error(err, kErrTimeout);
      return;
    }
    const uint8_t* rowp = R.slots + (size_t)s * R.P.slot_bytes + row_off;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int jb = 0; jb < NBW; ++jb) {
      if (jb < cnt) {
        const int b = warp + kMmaWarps * jb;
        const uint32_t cg = lds_u32(rowp + 16 * b);
        const uint32_t cu = lds_u32(rowp + up_off + 16 * b);
        const uint32_t bg = lds_u8(rowp + gs_off + b);
        const uint32_t bu = lds_u8(rowp + us_off + b);
        uint32_t hg0, hg1, hg2, hg3, hu0, hu1, hu2, hu3;
        e2m1x8_to_f16x2(cg, hg0, hg1, hg2, hg3);
        e2m1x8_to_f16x2(cu, hu0, hu1, hu2, hu3);
        float d[4];
        mma_16816_z(d, hg0, hu0, hg1, hu1, xb[jb][0], xb[jb][1]);
        mma_16816(d, hg2, hu2, hg3, hu3, xb[jb][2], xb[jb][3]);
        const float sg = e8m0_to_f32(bg), su = e8m0_to_f32(bu);
        acc[0] = fmaf(d[0], sg * xs0[jb], acc[0]);
        acc[1] = fmaf(d[1], sg * xs1[jb], acc[1]);
        acc[2] = fmaf(d[2], su * xs0[jb], acc[2]);
        acc[3] = fmaf(d[3], su * xs1[jb], acc[3]);
      }
    }
    float* dst = mypart + (size_t)s * (R.P.part_bytes / 4);
    if (!hand_over(R, j, s, ph, lane, warp, [&] {
          *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        })) {
      if (lane == 0) flag_error(err, kErrTimeout);
      return;
    }
    if (++s == R.S) {
      s = 0;
      ph ^= 1u;
    }
  }
}

template <class Kern, class... Args>
cudaError_t launch_ring(const DeviceInfo& di, Kern kern, int grid, int smem, cudaStream_t s,
                        bool pdl, Args... args) {
  cudaError_t e = ensure_smem(di, kern, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

cudaError_t launch_swiglu_mxfp4_mma(const uint8_t* packed, int n, int k, const uint16_t* x, int m,
                                    uint16_t* h, cudaStream_t s, bool pdl) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorNoDevice;
  if (m < 2 || m > 8 || k % 32 != 0) return cudaErrorInvalidConfiguration;
  const int nbw = (k / 32 + kMmaWarps - 1) / kMmaWarps;  // 32-blocks per consumer warp
  if (nbw > kMmaMaxNbw) return cudaErrorInvalidConfiguration;
  const MmaPlan one(k, 1);
  const int per_slot = one.slot_bytes + one.part_bytes + 24;
  int slots = TT_MMA_SMEM_BUDGET / per_slot;
  if (slots > TT_MMA_MAX_SLOTS) slots = TT_MMA_MAX_SLOTS;
  if (slots < 2) slots = 2;  // wide K: past the half-SM budget
  const MmaPlan plan(k, slots);
  if (plan.smem > di->smem_optin) return cudaErrorInvalidConfiguration;
  const int tiles = (n + kTileRows - 1) / kTileRows;
  const int grid = tiles < di->sms ? tiles : di->sms;
  switch (nbw) {
#define TT_MMA_CASE(NB)                                                                        \
  case NB:                                                                                     \
    return launch_ring(*di, swiglu_mxfp4_mma_kernel<NB>, grid, plan.smem, s, pdl, packed, n, k, \
                       m, x, h, slots, di->error_word);
    TT_MMA_CASE(1) TT_MMA_CASE(2) TT_MMA_CASE(3) TT_MMA_CASE(4) TT_MMA_CASE(5)
    TT_MMA_CASE(6) TT_MMA_CASE(7) TT_MMA_CASE(8) TT_MMA_CASE(9) TT_MMA_CASE(10)
#undef TT_MMA_CASE
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace tt
