// Tensor-core (tcgen05) MXFP4 gate/up SwiGLU for batches m = 4..64
// (k % 64 == 0; at m <= 8 only where its shared-memory plan fits).
//
// From a few batch rows on, the gate/up product is a dense contraction
// (config: Phi-4 sizes, K = 5120, N = 17920) whose cost on CUDA cores grows
// with m (one fp32 FMA per weight and batch row), so it runs on the
// 5th-generation tensor cores, where m = 4..16 cost the same.  The pages'
// prior art is Triton's tl.dot_scaled over the selected experts, with
// fast_math off because lossy accumulation broke the MoE trajectory
// (stardance.hackclub.com/projects/29750, MoE drift devlog); here the
// products are exact and accumulate in fp32 in tensor memory.
//
// Layout of the computation (swap-AB): one CTA owns 128 output rows (gate
// rows n0..n0+127 and the matching up rows) and all m batch rows.
//   A = W tile   [128 rows x 64 k]  f16 in tensor memory: row i in TMEM lane
//                                    i, two f16 of consecutive k per column
//   B = x tile   [N     x 64 k]     f16 in shared memory, K-major, 128-byte
//                                    swizzle, N = m rounded up to 16 (pad rows
//                                    are zero)
//   D_g, D_u     [128 x N] fp32 in tensor memory, in 2 or 4 accumulator sets
//                (the 4 k-steps of a k-tile go to the sets in turn, so
//                back-to-back MMAs do not wait on one accumulator)
// Warps 0-15 produce, in two groups of 8 that take the k-tiles in turn:
// thread t of a group decodes half a k-tile (one 32-weight block) of row
// t % 128 for gate and up: cvt.rn.f16x2.e2m1x2, then an exact HMUL2 by
// 2^(X_block - X_row) where X_row is the row's largest block exponent (so the
// f16 values stay in range and exact), stored with tcgen05.st into its row's
// TMEM lane; and converts its share of the x tile to f16 after an exact
// power-of-two prescale per x row that puts the row's largest |x| (over all
// of K, read once per CTA) in [2^14, 2^15), so no finite input leaves f16's
// range.  Warp 17 brings each k-tile in with three TMA loads (gate codes
// 128 x 32 B, up codes 128 x 32 B, both strided by the packed record size,
// and the x tile, whose padding rows TMA fills with zeros) into a ring of raw
// slots.  Warp 16 allocates tensor memory; warps 16 (gate) and 18 (up) wait
// for each stage and issue the tcgen05.mma (M=128, N, K=16, A from TMEM) x 4
// per matrix per stage, then tcgen05.commit releases the stage.  The 16
// producer warps finally read D with tcgen05.ld (warp w owns TMEM lanes
// 32(w%4)..+31 = rows and a quarter of the batch columns), add the
// accumulator sets in order, scale by 2^X_row and the postscale, apply
// silu(g)*u and store bf16.

#include "common.cuh"
#include "launch.h"
#include "layout.cuh"
#include "tensor_map.h"

namespace tt {
namespace {

#ifndef TT_TC_GROUP_WARPS
#define TT_TC_GROUP_WARPS 8
#endif
constexpr int kGroupWarps = TT_TC_GROUP_WARPS;  // one producer group: 8 warps = 256 threads
#ifndef TT_TC_GROUPS
#define TT_TC_GROUPS 2
#endif
constexpr int kGroups = TT_TC_GROUPS;            // groups decode k-tiles in turn
constexpr int kProdWarps = kGroupWarps * kGroups;
static_assert(kProdWarps == 16, "the epilogue splits the batch columns over 4 warp quads");
static_assert(kGroupWarps * 32 >= 128, "a producer group covers the tile's 128 rows");
constexpr int kMmaWarp = kProdWarps;             // tensor memory + the gate MMAs
constexpr int kTmaWarp = kProdWarps + 1;         // TMA loads
constexpr int kMmaWarpU = kProdWarps + 2;        // the up MMAs
constexpr int kThreads = (kProdWarps + 3) * 32;  // 608 with two groups
constexpr int kTileRows = 128;
constexpr int kTileK = 64;                      // f16: 128 bytes = one swizzle row
// Decoded stages and the most raw k-tiles in flight (4 stages fill the 512
// TMEM columns with the accumulator sets; 4 / 6 measured 45.1 / 57.3 us at
// m = 16 / 64 against 46.4 / 58.0 with 3 / 4, 8 raw slots no further gain).
#ifndef TT_TC_STAGES
#define TT_TC_STAGES 4
#endif
#ifndef TT_TC_MAX_RAW
#define TT_TC_MAX_RAW 6
#endif
constexpr int kStages = TT_TC_STAGES;  // decoded A/B stages
constexpr int kACol = 256;             // first TMEM column of the A tiles (after the D sets)
static_assert(kACol + 64 * kStages <= 512, "A stages fit the SM's 512 TMEM columns");
constexpr int kScaleBatch = 20;        // scale words per thread per load batch
constexpr int kScanDepth = 16;         // x-scan loads per lane in flight

// ---- tcgen05 / descriptor helpers ------------------------------------------
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (tcgen05 descriptor version 1).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);          // start address
  d |= uint64_t(1u) << 16;                        // leading byte offset (16 B; unused)
  d |= uint64_t((1024u >> 4) & 0x3FFFu) << 32;    // stride byte offset: 1024 B
  d |= uint64_t(1u) << 46;                        // descriptor version
  d |= uint64_t(2u) << 61;                        // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: A, B f16, D f32, both K-major.
__device__ __forceinline__ uint32_t idesc_f16(int n) {
  return (1u << 4)                        // D format f32
         | (0u << 7) | (0u << 10)         // A, B format f16
         | (uint32_t(n >> 3) << 17)       // N / 8
         | (uint32_t(kTileRows >> 4) << 24);  // M / 16
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D (+)= A B with A read from tensor memory (row i of A in TMEM lane i, two
// f16 of consecutive k per 32-bit column) and B from shared memory.
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 16 consecutive 32-bit columns of this warp's 32 TMEM lanes (thread i of
// the warp writes lane 32 (warp % 4) + i).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 4 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float* v) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// f16x2 (2^e, 2^e) for an exponent e <= 0; e < -24 underflows to zero.
__device__ __forceinline__ uint32_t pow2_f16x2(int e) {
  uint32_t h;
  if (e >= -14) h = uint32_t(e + 15) << 10;               // normal
  else if (e >= -24) h = 1u << (e + 24);                  // subnormal
  else h = 0u;
  return h | (h << 16);
}

// Physical offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte
// swizzled tile (8-row groups of 1024 bytes).
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return uint32_t(r) * 128u + (uint32_t(c ^ (r & 7)) << 4);
}

// 2-D TMA load of a box at (c0 inner, c1 outer) into shared memory,
// completion as tx bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Barrier among the producer warps only (warps 0 .. kProdWarps-1).
__device__ __forceinline__ void producer_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kProdWarps * 32) : "memory");
}

// Largest |x| of rows warp + kProdWarps i (i < NA) over all of K, into
// mx[i] (every lane): the rows' loads interleaved, kScanDepth per lane in
// flight.
template <int NA>
__device__ __forceinline__ void scan_x_rows(const uint16_t* __restrict__ x, int k, int warp,
                                            int lane, float* mx) {
  constexpr int kPer = kScanDepth / NA;  // chunks per row and lane per round trip
  const int nch = k >> 3;                // 16-byte chunks per row
  float a[NA];
#pragma unroll
  for (int i = 0; i < NA; ++i) a[i] = 0.f;
  for (int c0 = lane; c0 < nch; c0 += 32 * kPer) {
    uint4 v[NA][kPer];
#pragma unroll
    for (int i = 0; i < NA; ++i) {
      const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)(warp + kProdWarps * i) * k);
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int c = c0 + 32 * u;
        v[i][u] = c < nch ? __ldcg(xr + c) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int i = 0; i < NA; ++i)
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const uint32_t vw[4] = {v[i][u].x, v[i][u].y, v[i][u].z, v[i][u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          a[i] = fmaxf(a[i], fmaxf(fabsf(bf16_bits_to_f32(vw[e] & 0xFFFFu)),
                                   fabsf(bf16_bits_to_f32(vw[e] >> 16))));
      }
  }
#pragma unroll
  for (int i = 0; i < NA; ++i) mx[i] = warp_max(a[i]);
}

// Shared-memory plan of one CTA (offsets from a 1024-aligned base).
struct TcPlan {
  static constexpr int kMaxRaw = TT_TC_MAX_RAW;  // raw slots: packed k-tiles in flight
  int nraw;
  int np;          // MMA N (batch rows padded to 16)
  int nblk;        // k / 32
  int sstride;     // bytes per row of block scales in shared memory (odd word count)
  int stage_bytes; // one B (x) tile, 1024-aligned; the A tiles live in tensor memory
  int raw_bytes;   // one raw slot: gate 4 KB + up 4 KB + x np x 128 B
  int off_raw, off_scale, off_xr, off_sx, off_bar, off_tmem, total;
  __host__ __device__ TcPlan(int m, int k, int nraw_) : nraw(nraw_) {
    np = (m + 15) & ~15;
    nblk = k >> 5;
    sstride = 4 * ((nblk >> 1) | 1);
    stage_bytes = (np * 128 + 1023) & ~1023;
    raw_bytes = (2 * kTileRows * 32 + np * 128 + 127) & ~127;
    off_raw = kStages * stage_bytes;
    off_scale = off_raw + nraw * raw_bytes;
    off_xr = off_scale + kTileRows * sstride;
    off_sx = off_xr + 2 * kTileRows * 4;  // [64] x row maxima, [64] x row exponents
    off_bar = (off_sx + 2 * 64 * 4 + 7) & ~7;
    off_tmem = off_bar + (2 * kStages + 2 * kMaxRaw + 1) * 8;
    total = off_tmem + 16 + 1024;  // + alignment slack of the dynamic base
  }
};

__global__ void __launch_bounds__(kThreads, 1)
    tc_swiglu_kernel(const __grid_constant__ CUtensorMap map_w,
                     const __grid_constant__ CUtensorMap map_x, const uint8_t* __restrict__ packed,
                     const uint16_t* __restrict__ x, int n, int k, int m, int nraw,
                     uint16_t* __restrict__ h, int32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  const SwigluRecord L(k);
  const TcPlan P(m, k, nraw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (sbase - smem_u32(smem_raw));
  uint8_t* sscale = base + P.off_scale;  // [128 rows][gate nblk | up nblk], row stride sstride
  int* sxr = reinterpret_cast<int*>(base + P.off_xr);          // [2][128]
  uint32_t* xmax = reinterpret_cast<uint32_t*>(base + P.off_sx); // [64] max |x| bits per x row
  int* sxs = reinterpret_cast<int*>(xmax + 64);                  // [64] x row prescale exponents
  uint64_t* a_full = reinterpret_cast<uint64_t*>(base + P.off_bar);
  uint64_t* a_empty = a_full + kStages;
  uint64_t* raw_full = a_empty + kStages;
  uint64_t* raw_empty = raw_full + TcPlan::kMaxRaw;
  uint64_t* done = raw_empty + TcPlan::kMaxRaw;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + P.off_tmem);
  const int n0 = blockIdx.x * kTileRows;
  const int nkt = k / kTileK;
  // tensor memory: nacc independent accumulator sets, set j's D_g at column
  // 2 j np and D_u at (2 j + 1) np (2 nacc np <= 256); the decoded A tiles of
  // stage s at kACol + 64 s (gate 32 columns, then up 32).  The k-steps of a
  // k-tile go to the sets in turn, so consecutive MMAs never wait on each
  // other's accumulator; the epilogue adds the sets in a fixed order.
  const uint32_t tcols = 512u;
  const int nacc = P.np <= 32 ? 4 : 2;
  const uint32_t raw_tx = uint32_t(2 * kTileRows * 32 + P.np * 128);

  auto raw_slot = [&](int d) { return sbase + uint32_t(P.off_raw + d * P.raw_bytes); };
  const int pre = min(P.nraw, nkt);  // k-tiles requested before the main loop
  if (threadIdx.x == kTmaWarp * 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&a_full[s]), kGroupWarps * 32);
      mbar_init(smem_u32(&a_empty[s]), 2);  // one commit per MMA issuer
    }
    for (int d = 0; d < P.nraw; ++d) {
      mbar_init(smem_u32(&raw_full[d]), 1);
      mbar_init(smem_u32(&raw_empty[d]), kGroupWarps * 32);
    }
    mbar_init(smem_u32(done), 2);
    fence_mbar_init();
    // weights do not depend on the previous kernel: request the first
    // k-tiles while the CTA loads its block scales (x follows the wait)
    for (int kt = 0; kt < pre; ++kt) {
      const uint32_t dst = raw_slot(kt), bar = smem_u32(&raw_full[kt]);
      mbar_arrive_expect_tx(bar, raw_tx);
      tma_load_2d(dst, &map_w, kt * 32, n0, bar);
      tma_load_2d(dst + 4096, &map_w, k / 2 + kt * 32, n0, bar);
    }
  }
  if (warp == kMmaWarp) tmem_alloc(smem_u32(tmem_slot), tcols);
  if (threadIdx.x < 64) xmax[threadIdx.x] = 0u;
  // Block scales of the CTA's rows.  A record keeps a row's gate and up
  // scale bytes together (2 nblk bytes at a 16-byte aligned offset, a
  // multiple of 4), so all threads copy them as 32-bit words, each batch's
  // loads issued before its first store.  Rows past n read as zero.
  {
    const int nq = P.nblk >> 1;  // words per row
    const int total = kTileRows * nq;
    const int dr = kThreads / nq, dw = kThreads - dr * nq;  // index step in (row, word)
    int row = threadIdx.x / nq, wd = threadIdx.x - row * nq;
    for (int i0 = 0; i0 < total; i0 += kThreads * kScaleBatch) {
      uint32_t v[kScaleBatch];
      int lr = row, lw = wd;
#pragma unroll
      for (int i = 0; i < kScaleBatch; ++i) {
        const int idx = i0 + threadIdx.x + i * kThreads;
        v[i] = 0u;
        if (idx < total && n0 + lr < n)
          v[i] = __ldg(reinterpret_cast<const uint32_t*>(packed + (int64_t)(n0 + lr) * L.bytes +
                                                         L.gate_scales()) + lw);
        lw += dw;
        lr += dr;
        if (lw >= nq) {
          lw -= nq;
          ++lr;
        }
      }
#pragma unroll
      for (int i = 0; i < kScaleBatch; ++i) {
        const int idx = i0 + threadIdx.x + i * kThreads;
        if (idx < total) *reinterpret_cast<uint32_t*>(sscale + row * P.sstride + 4 * wd) = v[i];
        wd += dw;
        row += dr;
        if (wd >= nq) {
          wd -= nq;
          ++row;
        }
      }
    }
  }
  __syncthreads();
  // each row's largest block exponent (E8M0 255 is NaN and does not count):
  // gate rows by threads 0-127, up rows by 128-255
  if (threadIdx.x < 2 * kTileRows) {
    const int r = threadIdx.x & 127, which = threadIdx.x >> 7;
    const uint8_t* src = sscale + r * P.sstride + which * P.nblk;
    int emax = -1000;
    for (int b = 0; b < P.nblk; ++b) {
      const uint32_t sb = src[b];
      if (sb != 255u) emax = max(emax, int(sb) - 127);
    }
    sxr[which * kTileRows + r] = emax < -127 ? -127 : emax;
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  pdl_allow_next_grid();

  if (warp == kTmaWarp) {
    // ---------------- TMA loads ----------------
    if (lane == 0) {
      // (the first k-tiles' weights were requested in the prologue)
      pdl_wait_prior_grid();  // x is produced by the previous kernel
      for (int kt = 0; kt < pre; ++kt)
        tma_load_2d(raw_slot(kt) + 8192, &map_x, kt * kTileK, 0, smem_u32(&raw_full[kt]));
      bool ok = true;
      for (int kt = pre; kt < nkt; ++kt) {
        const int d = kt % P.nraw;
        ok = mbar_wait_bounded(smem_u32(&raw_empty[d]), uint32_t(((kt / P.nraw) - 1) & 1));
        if (!ok) break;
        const uint32_t dst = raw_slot(d), bar = smem_u32(&raw_full[d]);
        mbar_arrive_expect_tx(bar, raw_tx);
        tma_load_2d(dst, &map_w, kt * 32, n0, bar);
        tma_load_2d(dst + 4096, &map_w, k / 2 + kt * 32, n0, bar);
        tma_load_2d(dst + 8192, &map_x, kt * kTileK, 0, bar);
      }
      if (!ok) flag_error(err, kErrTimeout);
    }
    __syncwarp();
  } else if (warp == kMmaWarp || warp == kMmaWarpU) {
    // ---------------- MMA issuers: gate (kMmaWarp) and up (kMmaWarpU) ----
    // Two issuing threads, one per matrix: a thread issuing tcgen05.mma back
    // to back was the k-tile loop's pace (~40 ns an instruction).
    if (lane == 0) {
      const int mat = warp == kMmaWarpU ? 1 : 0;
      const uint32_t idesc = idesc_f16(P.np);
      bool ok = true;
      for (int kt = 0; kt < nkt && ok; ++kt) {
        const int s = kt % kStages;
        ok = mbar_wait_bounded(smem_u32(&a_full[s]), uint32_t((kt / kStages) & 1));
        if (!ok) break;
        fence_after_sync();
        // lane 0, the column of this matrix's A tile of stage s
        const uint32_t a = tmem + uint32_t(kACol + 64 * s + 32 * mat);
        const uint32_t bx = sbase + uint32_t(s * P.stage_bytes);
#pragma unroll
        for (int kk = 0; kk < kTileK / 16; ++kk) {
          const uint32_t koff = uint32_t(kk * 32);  // 16 f16 = 32 bytes along K
          const int j = kk % nacc;  // accumulator set
          const uint32_t acc = (kt > 0 || kk >= nacc) ? 1u : 0u;
          mma_f16_ta(tmem + uint32_t((2 * j + mat) * P.np), a + uint32_t(kk * 8),
                     smem_desc_sw128(bx + koff), idesc, acc);
        }
        mma_commit(smem_u32(&a_empty[s]));  // stage s free once both issuers' MMAs are done
      }
      if (!ok) flag_error(err, kErrTimeout);
      mma_commit(smem_u32(done));
      // Wait for both issuers' MMAs before tensor memory can be released.
      (void)mbar_wait_bounded(smem_u32(done), 0u);
    }
    __syncwarp();
  } else {
    // ---------------- producers: decode W, convert x ----------------
    // group g decodes k-tiles g, g + kGroups, ...; thread t of the group owns
    // part t / 128 of the k-tile (kPartK weights) of row t % 128
    constexpr int kParts = kGroupWarps * 32 / kTileRows;  // 2 (8 warps) or 1 (4 warps)
    constexpr int kPartK = kTileK / kParts;              // weights per part: 32 or 64
    constexpr int kPartWords = kPartK / 8;                // 32-bit code words per part
    static_assert(kPartWords == 4 || kPartWords == 8, "a part is 16 or 32 TMEM columns");
    const int g = warp / kGroupWarps;
    const int t = threadIdx.x - g * kGroupWarps * 32, r = t & 127, part = t >> 7;
    const int xg = sxr[r], xu = sxr[kTileRows + r];
    // Each x row gets the exact power-of-two prescale 2^sxs[i] that puts its
    // largest |x| over the whole row in [2^14, 2^15): every finite value then
    // fits f16 and keeps its bits down to 2^-28 of the row's max.  The
    // producer warps scan x once (all of K) after the dependency wait; the
    // epilogue divides the factor back out.
    pdl_wait_prior_grid();  // x is produced by the previous kernel
    {
      // Warp w scans its x rows (w, w + 16, w + 32, w + 48 below m) together,
      // kScanDepth loads per lane in flight across them: two round trips per
      // 5120-wide row at m <= 16, five for four rows at m = 64 (row by row,
      // four loads at a time, it was twenty, ~10 us).
      const int na = warp < m ? min(4, (m - warp + kProdWarps - 1) / kProdWarps) : 0;
      float mxr[4] = {0.f, 0.f, 0.f, 0.f};
      switch (na) {
        case 1: scan_x_rows<1>(x, k, warp, lane, mxr); break;
        case 2: scan_x_rows<2>(x, k, warp, lane, mxr); break;
        case 3: scan_x_rows<3>(x, k, warp, lane, mxr); break;
        case 4: scan_x_rows<4>(x, k, warp, lane, mxr); break;
        default: break;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = warp + kProdWarps * i;
        if (lane == 0 && row < P.np) xmax[row] = __float_as_uint(mxr[i]);
      }
    }
    producer_bar_sync();
    if (threadIdx.x < P.np) {
      const float mx = __uint_as_float(xmax[threadIdx.x]);
      sxs[threadIdx.x] = mx > 0.f ? min(f16_prescale_exponent(mx), 127) : 0;
    }
    producer_bar_sync();
    bool ok = true;
    for (int kt = g; kt < nkt; kt += kGroups) {
      const int s = kt % kStages, d = kt % P.nraw;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&raw_full[d]),
                                                     uint32_t((kt / P.nraw) & 1)));
      if (!ok) break;
      const uint8_t* rw = base + P.off_raw + d * P.raw_bytes;
      // Every load of the k-tile first, into registers: the stores below go
      // to the same shared memory, so they would otherwise hold each later
      // load back.  Only the stores wait for the stage to be free.  The raw
      // slot is released after the stores, which consume every loaded value,
      // so no copy into the slot can overtake a load from it.
      constexpr int kPB = (kPartK + 31) / 32;  // 32-blocks per part
      uint32_t w[2][kPartWords], sb[2][kPB];
#pragma unroll
      for (int mat = 0; mat < 2; ++mat) {
        const uint8_t* src = rw + mat * 4096 + r * 32 + part * (kPartK / 2);
        if constexpr (kPartWords == 8) {
          const uint4 c0 = *reinterpret_cast<const uint4*>(src);
          const uint4 c1 = *reinterpret_cast<const uint4*>(src + 16);
          w[mat][0] = c0.x;
          w[mat][1] = c0.y;
          w[mat][2] = c0.z;
          w[mat][3] = c0.w;
          w[mat][4] = c1.x;
          w[mat][5] = c1.y;
          w[mat][6] = c1.z;
          w[mat][7] = c1.w;
        } else if constexpr (kPartWords == 4) {
          const uint4 c = *reinterpret_cast<const uint4*>(src);
          w[mat][0] = c.x;
          w[mat][1] = c.y;
          w[mat][2] = c.z;
          w[mat][3] = c.w;
        } else {
          const uint2 c = *reinterpret_cast<const uint2*>(src);
          w[mat][0] = c.x;
          w[mat][1] = c.y;
        }
#pragma unroll
        for (int pb = 0; pb < kPB; ++pb)
          sb[mat][pb] = sscale[r * P.sstride + mat * P.nblk + kt * 2 + (part * kPartK) / 32 + pb];
      }
      constexpr int kXJ = 64 * 8 / (kGroupWarps * 32);  // x pieces per thread (np <= 64)
      uint4 xv[kXJ];
      int xe[kXJ];
#pragma unroll
      for (int j = 0; j < kXJ; ++j) {
        const int c = t + j * kGroupWarps * 32;  // row c / 8, 16-byte piece c % 8
        const int row = c >> 3, piece = c & 7;
        xv[j] = make_uint4(0u, 0u, 0u, 0u);
        xe[j] = 0;
        if (row < P.np) {
          xv[j] = *reinterpret_cast<const uint4*>(rw + 8192 + row * 128 + piece * 16);
          xe[j] = sxs[row];
        }
      }
      if (kt >= kStages)
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&a_empty[s]),
                                                       uint32_t(((kt / kStages) - 1) & 1)));
      if (!ok) break;
      fence_after_sync();  // the stage's MMAs (committed) are done with its A columns
      uint8_t* stage = base + s * P.stage_bytes;  // the B (x) tile
      // W: kPartK weights per matrix -> kPartK / 2 f16x2 columns of this row's
      // TMEM lane (k = kPartK part .. kPartK (part + 1) - 1 of the k-tile, two
      // per column), each code word scaled by its own 32-block's factor
      const uint32_t arow =
          tmem + (uint32_t(r & ~31) << 16) + uint32_t(kACol + 64 * s + (kPartK / 2) * part);
#pragma unroll
      for (int mat = 0; mat < 2; ++mat) {
        uint32_t av[4 * kPartWords];
#pragma unroll
        for (int q = 0; q < kPartWords; ++q) {
          const uint32_t sbq = sb[mat][q / 4];  // 4 code words per 32-block
          const uint32_t f =
              sbq == 255u ? 0x7E007E00u : pow2_f16x2(int(sbq) - 127 - (mat ? xu : xg));
          uint32_t h0, h1, h2, h3;
          e2m1x8_to_f16x2(w[mat][q], h0, h1, h2, h3);
          av[4 * q + 0] = hmul2(h0, f);
          av[4 * q + 1] = hmul2(h1, f);
          av[4 * q + 2] = hmul2(h2, f);
          av[4 * q + 3] = hmul2(h3, f);
        }
#pragma unroll
        for (int h = 0; h < kPartWords / 4; ++h)
          tmem_st16(arow + uint32_t(32 * mat + 16 * h), av + 16 * h);
      }
      tmem_wait_st();
      // x: bf16 * 2^sxs[row] -> f16, within range by the choice of sxs
#pragma unroll
      for (int j = 0; j < kXJ; ++j) {
        const int c = t + j * kGroupWarps * 32;
        const int row = c >> 3, piece = c & 7;
        if (row < P.np) {
          const uint32_t vw[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
          const float two_s = scalbnf(1.0f, xe[j]);
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[e] = pack_f16x2_scaled(bf16_bits_to_f32(vw[e] & 0xFFFFu),
                                     bf16_bits_to_f32(vw[e] >> 16), two_s);  // exact
          *reinterpret_cast<uint4*>(stage + sw128(row, piece)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      fence_proxy_async();  // x stores -> the MMA's shared-memory reads
      fence_before_sync();  // A stores -> the MMA
      mbar_arrive(smem_u32(&a_full[s]));
      mbar_arrive(smem_u32(&raw_empty[d]));
    }
    if (!ok) flag_error(err, kErrTimeout);
  }

  // ---------------- epilogue: the 16 producer warps ----------------
  // Warp w reads TMEM lanes 32 (w % 4) .. + 31 (its rows, thread = row) and
  // the w / 4-th quarter of the batch columns, 4 columns per load (one warp
  // quad per column quarter: at m = 64 the 4-warp epilogue took ~9 us).
  if (warp < kProdWarps) {
    const int q = warp & 3, cq = warp >> 2;
    const int r = q * 32 + lane;
    const bool ok = mbar_wait_bounded(smem_u32(done), 0u);
    fence_after_sync();
    if (ok) {
      pdl_wait_prior_grid();  // (no-op if already waited) before writing h
      const int nr = n0 + r;
      const uint8_t* rec = packed + (int64_t)(nr < n ? nr : 0) * L.bytes;
      const float pg = *reinterpret_cast<const float*>(rec + L.post);
      const float pu = *reinterpret_cast<const float*>(rec + L.post + 4);
      const int eg = sxr[r], eu = sxr[kTileRows + r];
      const uint32_t lane_base = uint32_t(q * 32) << 16;
      const int cpq = P.np / (kProdWarps / 4);  // columns per quarter (np % 16 == 0)
      for (int c0 = cq * cpq; c0 < (cq + 1) * cpq; c0 += 4) {
        float g[4], u[4];
        tmem_ld4(tmem + lane_base + uint32_t(c0), g);
        tmem_ld4(tmem + lane_base + uint32_t(P.np + c0), u);
        for (int j = 1; j < nacc; ++j) {  // the other accumulator sets, in order
          float gj[4], uj[4];
          tmem_ld4(tmem + lane_base + uint32_t(2 * j * P.np + c0), gj);
          tmem_ld4(tmem + lane_base + uint32_t((2 * j + 1) * P.np + c0), uj);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            g[i] += gj[i];
            u[i] += uj[i];
          }
        }
        if (nr < n) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int mm = c0 + i;
            if (mm < m) {
              // exact power-of-two factors: the row's block exponent and the
              // x row's prescale, folded into the postscale
              const float sg = scalbnf(pg, eg - sxs[mm]), su = scalbnf(pu, eu - sxs[mm]);
              __nv_bfloat16 b = __float2bfloat16_rn(silu_mul(g[i] * sg, u[i] * su));
              h[(size_t)mm * n + nr] = *reinterpret_cast<uint16_t*>(&b);
            }
          }
        }
      }
    } else if (lane == 0) {
      flag_error(err, kErrTimeout);
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    fence_after_sync();
    tmem_dealloc(tmem, tcols);
  }
}

}  // namespace

// Deepest raw ring (most k-tiles of packed weights in flight) that fits.
static int pick_nraw(int m, int k, int limit) {
  for (int r = TcPlan::kMaxRaw; r >= 2; --r)
    if (TcPlan(m, k, r).total <= limit) return r;
  return 0;
}

int tc_swiglu_smem_bytes(int m, int k) { return TcPlan(m, k, 2).total; }

cudaError_t launch_swiglu_mxfp4_tc(const uint8_t* packed, int n, int k, const uint16_t* x, int m,
                                   uint16_t* h, cudaStream_t s, bool pdl) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorNoDevice;
  if (k % kTileK != 0 || m < 1 || m > 64) return cudaErrorInvalidConfiguration;
  const int nraw = pick_nraw(m, k, di->smem_optin);
  if (nraw == 0) return cudaErrorInvalidConfiguration;
  const TcPlan P(m, k, nraw);
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const SwigluRecord L(k);
  CUtensorMap map_w, map_x;
  {
    const cuuint64_t dims[2] = {cuuint64_t(L.bytes), cuuint64_t(n)};
    const cuuint64_t strides[1] = {cuuint64_t(L.bytes)};
    const cuuint32_t box[2] = {32u, cuuint32_t(kTileRows)};
    const cuuint32_t estr[2] = {1u, 1u};
    if (enc(&map_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(packed), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {cuuint64_t(k), cuuint64_t(m)};
    const cuuint64_t strides[1] = {cuuint64_t(k) * 2};
    const cuuint32_t box[2] = {cuuint32_t(kTileK), cuuint32_t(P.np)};
    const cuuint32_t estr[2] = {1u, 1u};
    if (enc(&map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t e = ensure_smem(*di, tc_swiglu_kernel, P.total);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n + kTileRows - 1) / kTileRows);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = P.total;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tc_swiglu_kernel, map_w, map_x, packed, x, n, k, m, nraw, h,
                            di->error_word);
}

}  // namespace tt
