// MXFP4 building blocks shared by the dense and MoE matvec kernels: the
// 32-weight E2M1 dot product, the per-warp bulk-copy ring, warp reductions
// and the batched SwiGLU epilogue.
#pragma once

#include "common.cuh"

namespace tt {

// 32 E2M1 codes (one 16-byte chunk) dotted with 32 f16 values (16 f16x2),
// fp32 accumulation in four chains.
__device__ __forceinline__ float dot32(const uint4& c, const uint32_t* xv) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  uint32_t h[16];
  e2m1x8_to_f16x2(c.x, h[0], h[1], h[2], h[3]);
  e2m1x8_to_f16x2(c.y, h[4], h[5], h[6], h[7]);
  e2m1x8_to_f16x2(c.z, h[8], h[9], h[10], h[11]);
  e2m1x8_to_f16x2(c.w, h[12], h[13], h[14], h[15]);
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    fma_f16x2_f32(a0, a1, h[i], xv[i]);
    fma_f16x2_f32(a2, a3, h[i + 1], xv[i + 1]);
  }
  return (a0 + a1) + (a2 + a3);
}

__device__ __forceinline__ void decode32(const uint4& c, uint32_t* h) {
  e2m1x8_to_f16x2(c.x, h[0], h[1], h[2], h[3]);
  e2m1x8_to_f16x2(c.y, h[4], h[5], h[6], h[7]);
  e2m1x8_to_f16x2(c.z, h[8], h[9], h[10], h[11]);
  e2m1x8_to_f16x2(c.w, h[12], h[13], h[14], h[15]);
}

__device__ __forceinline__ float dot32_decoded(const uint32_t* h, const uint32_t* xv) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    fma_f16x2_f32(a0, a1, h[i], xv[i]);
    fma_f16x2_f32(a2, a3, h[i + 1], xv[i + 1]);
  }
  return (a0 + a1) + (a2 + a3);
}

// D = A * B + D for one mma.sync m16n8k16 tile, f16 inputs, fp32 accumulators
// (the warp-level tensor-core instruction).  Not volatile: a pure function of
// its registers, free to be scheduled.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D = A * B.
__device__ __forceinline__ void mma_16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

// Per-warp ring of bulk-copy slots.  Item j of the warp is a "unit" of up to
// `rpc` consecutive records starting at record first(j); one bulk copy
// brings the whole unit into slot j % slots.  Items are consumed in order:
// the ring tracks the slot and mbarrier parity of the next one (no integer
// division on the per-record path).
struct WarpRing {
  uint8_t* base;
  uint64_t* bars;
  int slots;
  int slot_bytes;     // rpc * record bytes
  int rec_bytes;
  const uint8_t* packed;
  uint64_t policy;
  int cur = 0;           // slot of the next item to consume
  uint32_t phase = 0;    // mbarrier parity of that item

  __device__ void init(int lane) {
    if (lane == 0) {
      for (int s = 0; s < slots; ++s) mbar_init(smem_u32(&bars[s]), 1);
      fence_mbar_init();
    }
    __syncwarp();
  }
  // lane 0 only: copy `count` records starting at record `first` into slot s.
  __device__ void issue_to(int s, int first, int count) {
    const uint32_t bar = smem_u32(&bars[s]);
    const uint32_t bytes = uint32_t(count * rec_bytes);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(smem_u32(base + (size_t)s * slot_bytes), packed + (int64_t)first * rec_bytes, bytes,
             bar, policy);
  }
  // The next item's slot once its copy has landed, nullptr after a timeout
  // (warp-uniform).  Refill that slot with issue_to(cur, ...), then advance().
  __device__ const uint8_t* wait_next() {
    const bool ok = mbar_wait_bounded(smem_u32(&bars[cur]), phase);
    if (!__all_sync(0xffffffffu, ok)) return nullptr;
    return base + (size_t)cur * slot_bytes;
  }
  __device__ void advance() {
    if (++cur == slots) {
      cur = 0;
      phase ^= 1u;
    }
  }
  // After a timeout at item j: give the copies already issued a bounded
  // chance to land before the CTA may exit.
  __device__ void drain(int j, int nitems) {
    const int issued = min(nitems, j + slots);
    for (int t = j + 1; t < issued; ++t)
      (void)mbar_wait_bounded(smem_u32(&bars[t % slots]), uint32_t((t / slots) & 1));
  }
};

// Sums four values over the warp in six shuffles.  Lanes 0-7 get the total
// of a, 8-15 of b, 16-23 of c, 24-31 of d.
__device__ __forceinline__ float warp_sum4(float a, float b, float c, float d, int lane) {
  const bool hi16 = (lane & 16) != 0;
  float k0 = hi16 ? c : a, k1 = hi16 ? d : b;
  const float s0 = hi16 ? a : c, s1 = hi16 ? b : d;
  k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
  k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
  const bool hi8 = (lane & 8) != 0;
  float k = hi8 ? k1 : k0;
  const float s = hi8 ? k0 : k1;
  k += __shfl_xor_sync(0xffffffffu, s, 8);
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  return k;
}

// The SwiGLU epilogue of a warp's records, batched: lane (t % 32) keeps the
// postscaled g and u of the warp's t-th record, and every 32 records (or at
// the end) all lanes apply silu(g)*u and store bf16 together, instead of one
// lane per record.
struct EpilogueBatch {
  float g = 0.f, u = 0.f;
  int row = -1;
  int fill = 0;

  // v holds a reduced value on every lane; gsrc/usrc are lanes holding this
  // record's g and u sums.
  __device__ void put(float v, int gsrc, int usrc, float pg, float pu, float inv, int r,
                      int lane) {
    const float gg = __shfl_sync(0xffffffffu, v, gsrc);
    const float uu = __shfl_sync(0xffffffffu, v, usrc);
    if (lane == fill) {
      g = gg * inv * pg;
      u = uu * inv * pu;
      row = r;
    }
    ++fill;
  }
  __device__ void flush(uint16_t* __restrict__ h) {
    if (row >= 0) h[row] = f32_to_bf16_rne(silu_mul(g, u));
    row = -1;
    fill = 0;
  }
};

}  // namespace tt
