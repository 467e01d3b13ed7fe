// Single-token grouped-query attention over a bf16 KV cache: the attention of
// one decode step.
//
// Method: ThinTensor Dev Log #3 "SmolLM3-3B Results" (the kernel side of the
// quality profile): attention is single-token GQA; query head h reads kv head
// h // (heads // kv_heads) and scores each cached key as sum(key * q) *
// scale; the KV cache stays bf16 ("KV cache: BF16", causal KV).  The project
// page's "What I've Done", item 3, unrolls that kernel over a fixed token
// bucket; here the context length is a runtime value and nothing is
// unrolled over it.
//
//   o[h] = sum_{t < len} softmax_t(scale * q[h] . k[j][t]) * v[j][t],
//   j = h / (heads / kv_heads)
//
// The G = heads / kv_heads query heads of one kv head share every K and V
// row, so the two products are small dense contractions and run on mma.sync
// (m16n8k16, bf16 in, fp32 accumulate):
//   scores  S[token][head] = K[token][:] . Q[head][:]   A = K (16 tokens x 16
//           dims, straight from the cache rows), B = Q^T (8 heads);
//   output  O^T[dim][head] += V^T[dim][token] P^T[token][head]   A = V^T
//           (16 dims x 16 tokens, paired from two cache rows with byte
//           permutes), B = P^T (the softmax weights, moved from the score
//           fragments' layout with four shuffles per 16 tokens).
// The weights P are split into bf16 hi + lo parts (p = hi + lo to ~2^-17
// relative), so the P.V product keeps fp32-level accuracy; the scores are
// exact bf16 x bf16 products summed in fp32.
//
// Work layout ("split the tokens"): grid (S splits, kv_heads), 4 warps per
// CTA, one CTA per SM.  A CTA takes a contiguous range of tiles (64 tokens
// for head_dim 64, 32 for head_dim 128: 16 KB of K and V either way) of one
// kv head; its warps take every 4th tile, each with its own ring of
// shared-memory stages and an mbarrier per stage.  A stage is filled by TMA
// tensor copies of a tile's tokens x 64 dims (128 bytes a row, 128-byte
// swizzle, so the fragment loads are free of bank conflicts); the tensor
// maps end at len, so rows past the end arrive as zeros and the cache beyond
// len is never read.  Before waiting for the preceding kernel, each warp
// prefetches its first tiles into L2.  Each warp keeps an online softmax
// (running max, sum and output in
// log2 units); the CTA merges its warps and writes one partial (max, sum,
// unnormalised output per head) to the caller's workspace.  A second kernel,
// launched programmatically behind the first, merges the S partials of each
// query head in a fixed order, normalises and rounds to bf16.
#include <cmath>

#include "common.cuh"
#include "launch.h"
#include "mxfp4_core.cuh"
#include "tensor_map.h"

namespace tt {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kMergeThreads = 256;
constexpr int kMergeBatch = 8;  // split partials one merge thread loads at once
constexpr uint32_t kFull = 0xffffffffu;

// A tile is kTok tokens; its K and V rows arrive as TMA boxes of kTok
// tokens x 64 dims (128-byte rows); a stage is 16 KB either way.
template <int D>
struct AttnPlan {
  static constexpr int kTok = D == 64 ? 64 : 32;  // tokens per tile
  static constexpr int kBox = kTok * 128;         // one TMA box
  static constexpr int kCh = D / 64;              // boxes per token range
  static constexpr int kStage = 2 * kCh * kBox;   // K boxes, then V boxes
  static constexpr int kStages = 3;
  static constexpr int kRing = kWarps * kStages * kStage;
  static constexpr int kSmem = 1024 + kRing + kWarps * kStages * 8;  // + 1024-byte alignment
};

// Floats per split partial: O [G][D], then max [G], then sum [G]; padded to
// 16 bytes.
__host__ __device__ constexpr int partial_floats(int G, int D) { return (G * (D + 2) + 3) & ~3; }

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// TMA tensor copy of one box at (x = dim, y = token, z = kv head).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// L2 prefetch of one box (no shared-memory destination, no completion).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

// Byte offset of 16-byte chunk c of row r in a box written with the 128-byte
// swizzle (chunk index XOR row mod 8; boxes start 1024-byte aligned).
__device__ __forceinline__ int swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// (a, b) -> bf16x2 with a in the low half, round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Selects the low (h = 0) or high (h = 1) bf16 halves of a and b into one
// pair, a's in the low half.
__device__ __forceinline__ uint32_t pair_halves(uint32_t a, uint32_t b, int h) {
  return __byte_perm(a, b, h ? 0x7632 : 0x5410);
}

// The 16-byte piece of a row that lane quad position qd reads for 32-dim
// chunk c of the score contraction: pieces 2qd (+1 for odd c); with the
// swizzle the eight lanes of one shared-memory phase hit eight different
// bank groups.
__device__ __forceinline__ int score_piece(int c, int qd) { return 8 * (c >> 1) + 2 * qd + (c & 1); }

template <int D, int NH>
__global__ void __launch_bounds__(kThreads, 1)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const uint16_t* __restrict__ q,
                      int G, int64_t len, float sl2, float* __restrict__ part0,
                      int32_t* __restrict__ err) {
  using P = AttnPlan<D>;
  constexpr int KC = D / 32;  // 32-dim chunks of the score contraction
  constexpr int MT = D / 16;  // 16-dim tiles of the output
  constexpr int kTok = P::kTok, kBox = P::kBox;
  constexpr int TM = kTok / 16;  // 16-token tiles of the scores
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, qd = lane & 3;
  const int s = blockIdx.x, S = gridDim.x, j = blockIdx.y;
  const int PS = partial_floats(G, D);
  const int64_t T = (len + kTok - 1) / kTok;
  const int64_t tb = T * s / S, te = T * (s + 1) / S;  // this CTA's tiles (at least one)
  const int mine = te - tb > warp ? int((te - tb - warp + kWarps - 1) / kWarps) : 0;
  uint8_t* ring = smem + warp * (P::kStages * P::kStage);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P::kRing) + warp * P::kStages;

  if (lane == 0) {
    for (int i = 0; i < P::kStages; ++i) mbar_init(smem_u32(&bars[i]), 1);
    fence_mbar_init();
    prefetch_tensor_map(&tmk);
    prefetch_tensor_map(&tmv);
  }
  __syncwarp();
  pdl_allow_next_grid();
  // While the preceding kernel finishes: pull the warp's first tiles into L2.
  // L2 is where every write lands, so rows that kernel still appends are
  // read fresh by the copies below, which start after the wait.
  if (lane == 0)
    for (int i = 0; i < mine && i < P::kStages; ++i) {
      const int t0 = int((tb + warp + int64_t(kWarps) * i) * kTok);
#pragma unroll
      for (int h = 0; h < P::kCh; ++h) {
        tma_prefetch_3d(&tmk, 64 * h, t0, j);
        tma_prefetch_3d(&tmv, 64 * h, t0, j);
      }
    }
  pdl_wait_prior_grid();  // q and the newest cache rows come from earlier kernels

  const uint64_t pol = l2_evict_first_policy();
  // The warp's i-th tile (tile tb + warp + 4i) into stage i % kStages; rows
  // past len arrive as zeros (their weights are zero too).
  auto issue = [&](int i) {
    const int st = i % P::kStages;
    const int t0 = int((tb + warp + int64_t(kWarps) * i) * kTok);
    const uint32_t kd = smem_u32(ring + st * P::kStage), bar = smem_u32(&bars[st]);
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, uint32_t(P::kStage));
#pragma unroll
      for (int h = 0; h < P::kCh; ++h) {
        tma_load_3d(kd + h * kBox, &tmk, 64 * h, t0, j, bar, pol);
        tma_load_3d(kd + (P::kCh + h) * kBox, &tmv, 64 * h, t0, j, bar, pol);
      }
    }
  };
  for (int i = 0; i < mine && i < P::kStages; ++i) issue(i);

  // Q^T as the B operand of the score mma: lane (g, qd) holds head g + 8 nh,
  // the pieces score_piece(c, qd); zero past G.
  uint4 qf[NH][KC];
#pragma unroll
  for (int nh = 0; nh < NH; ++nh) {
    const int h = g + 8 * nh;
#pragma unroll
    for (int c = 0; c < KC; ++c)
      qf[nh][c] = h < G ? __ldcg(reinterpret_cast<const uint4*>(
                              q + (int64_t(j) * G + h) * D + 8 * score_piece(c, qd)))
                        : make_uint4(0u, 0u, 0u, 0u);
  }

  // Online softmax state for the lane's heads 8 nh + 2qd + {0, 1} (log2
  // units) and O^T fragments: o[nh][mt] = (dim row g | g + 8) x (head 2qd,
  // 2qd + 1).
  float mrun[NH][2], lsum[NH][2];
  float o[NH][MT][4];
#pragma unroll
  for (int nh = 0; nh < NH; ++nh) {
    mrun[nh][0] = mrun[nh][1] = -INFINITY;
    lsum[nh][0] = lsum[nh][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) o[nh][mt][0] = o[nh][mt][1] = o[nh][mt][2] = o[nh][mt][3] = 0.f;
  }

  for (int i = 0; i < mine; ++i) {
    const int st = i % P::kStages;
    const uint32_t ph = uint32_t((i / P::kStages) & 1);
    if (!__all_sync(kFull, mbar_wait_bounded(smem_u32(&bars[st]), ph))) {
      if (lane == 0) flag_error(err, kErrTimeout);
      // let the copies still in flight land before the ring is reused
      for (int i2 = i; i2 < mine && i2 < i + P::kStages; ++i2)
        (void)mbar_wait_bounded(smem_u32(&bars[i2 % P::kStages]),
                                uint32_t((i2 / P::kStages) & 1));
#pragma unroll
      for (int nh = 0; nh < NH; ++nh) {  // this warp contributes nothing
        mrun[nh][0] = mrun[nh][1] = -INFINITY;
        lsum[nh][0] = lsum[nh][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
          o[nh][mt][0] = o[nh][mt][1] = o[nh][mt][2] = o[nh][mt][3] = 0.f;
      }
      break;
    }
    const uint8_t* kd = ring + st * P::kStage;
    const uint8_t* vd = kd + P::kCh * kBox;
    const int64_t t0 = (tb + warp + int64_t(kWarps) * i) * kTok;
    const int nt = len - t0 < kTok ? int(len - t0) : kTok;

    // scores sc[tm][nh]: tokens 16 tm + (g | g + 8) x heads 8 nh + 2qd + (0 | 1)
    float sc[TM][NH][4];
#pragma unroll
    for (int tm = 0; tm < TM; ++tm) {
#pragma unroll
      for (int nh = 0; nh < NH; ++nh)
        sc[tm][nh][0] = sc[tm][nh][1] = sc[tm][nh][2] = sc[tm][nh][3] = 0.f;
      const int r0 = 16 * tm + g, r1 = r0 + 8;
#pragma unroll
      for (int c = 0; c < KC; ++c) {
        const int p = score_piece(c, qd);
        const uint8_t* box = kd + (p >> 3) * kBox;
        const uint4 a = *reinterpret_cast<const uint4*>(box + swz(r0, p & 7));
        const uint4 b = *reinterpret_cast<const uint4*>(box + swz(r1, p & 7));
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) {
          mma_bf16(sc[tm][nh], a.x, b.x, a.y, b.y, qf[nh][c].x, qf[nh][c].y);
          mma_bf16(sc[tm][nh], a.z, b.z, a.w, b.w, qf[nh][c].z, qf[nh][c].w);
        }
      }
    }
    // scale to log2 units, mask tokens past the end, per-head tile max
#pragma unroll
    for (int nh = 0; nh < NH; ++nh) {
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int tm = 0; tm < TM; ++tm) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = 16 * tm + g + 8 * (e >> 1);
          const float v = tok < nt ? sc[tm][nh][e] * sl2 : -INFINITY;
          sc[tm][nh][e] = v;
          mx[e & 1] = fmaxf(mx[e & 1], v);
        }
      }
      float alpha[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float m = mx[h];
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 8));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 16));
        const float mn = fmaxf(mrun[nh][h], m);  // finite: the tile has a token
        alpha[h] = exp2f(mrun[nh][h] - mn);      // 0 on the first tile
        mrun[nh][h] = mn;
      }
#pragma unroll
      for (int tm = 0; tm < TM; ++tm) {
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[tm][nh][e] = exp2f(sc[tm][nh][e] - mrun[nh][e & 1]);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float t = 0.f;
#pragma unroll
        for (int tm = 0; tm < TM; ++tm) t += sc[tm][nh][h] + sc[tm][nh][h + 2];
        lsum[nh][h] = lsum[nh][h] * alpha[h] + t;
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        o[nh][mt][0] *= alpha[0];
        o[nh][mt][1] *= alpha[1];
        o[nh][mt][2] *= alpha[0];
        o[nh][mt][3] *= alpha[1];
      }
    }

    // O^T += V^T P^T, one 16-token chunk (= score tile tm) at a time
    const int src0 = 4 * (2 * qd) + (g >> 1), src1 = src0 + 4;  // lanes holding tokens 2qd, 2qd+1
#pragma unroll
    for (int tm = 0; tm < TM; ++tm) {
      // P^T fragments (hi and lo) for head 8 nh + g, tokens 2qd, 2qd + 1 (b0)
      // and 2qd + 8, 2qd + 9 (b1) of this chunk
      uint32_t bh[NH][2], bl[NH][2];
#pragma unroll
      for (int nh = 0; nh < NH; ++nh) {
        const float* c = sc[tm][nh];
        const uint32_t h0 = pack_bf16x2(c[0], c[1]), h1 = pack_bf16x2(c[2], c[3]);
        const uint32_t l0 = pack_bf16x2(c[0] - __uint_as_float(h0 << 16),
                                        c[1] - __uint_as_float(h0 & 0xFFFF0000u));
        const uint32_t l1 = pack_bf16x2(c[2] - __uint_as_float(h1 << 16),
                                        c[3] - __uint_as_float(h1 & 0xFFFF0000u));
        const int hf = g & 1;
        bh[nh][0] = pair_halves(__shfl_sync(kFull, h0, src0), __shfl_sync(kFull, h0, src1), hf);
        bh[nh][1] = pair_halves(__shfl_sync(kFull, h1, src0), __shfl_sync(kFull, h1, src1), hf);
        bl[nh][0] = pair_halves(__shfl_sync(kFull, l0, src0), __shfl_sync(kFull, l0, src1), hf);
        bl[nh][1] = pair_halves(__shfl_sync(kFull, l1, src0), __shfl_sync(kFull, l1, src1), hf);
      }
      // V rows 2qd, 2qd + 1, 2qd + 8, 2qd + 9 of the chunk; 16-byte piece g
      // (dims 8g..8g+7) and, for D = 128, piece g + 8 (dims 64 + 8g..)
      constexpr int CH = P::kCh;
      const int rv = 16 * tm + 2 * qd;
      uint4 v[4][CH];
#pragma unroll
      for (int ch = 0; ch < CH; ++ch) {
        const uint8_t* box = vd + ch * kBox;
        v[0][ch] = *reinterpret_cast<const uint4*>(box + swz(rv, g));
        v[1][ch] = *reinterpret_cast<const uint4*>(box + swz(rv + 1, g));
        v[2][ch] = *reinterpret_cast<const uint4*>(box + swz(rv + 8, g));
        v[3][ch] = *reinterpret_cast<const uint4*>(box + swz(rv + 9, g));
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        // dim rows of tile mt: D = 64: row g -> 8g + 2mt, row g + 8 -> 8g + 2mt + 1;
        // D = 128: row g -> 8g + mt, row g + 8 -> 64 + 8g + mt
        uint32_t a0, a1, a2, a3;
        if constexpr (D == 64) {
          a0 = pair_halves(word(v[0][0], mt), word(v[1][0], mt), 0);
          a1 = pair_halves(word(v[0][0], mt), word(v[1][0], mt), 1);
          a2 = pair_halves(word(v[2][0], mt), word(v[3][0], mt), 0);
          a3 = pair_halves(word(v[2][0], mt), word(v[3][0], mt), 1);
        } else {
          const int w = mt >> 1, hf = mt & 1;
          a0 = pair_halves(word(v[0][0], w), word(v[1][0], w), hf);
          a1 = pair_halves(word(v[0][CH - 1], w), word(v[1][CH - 1], w), hf);
          a2 = pair_halves(word(v[2][0], w), word(v[3][0], w), hf);
          a3 = pair_halves(word(v[2][CH - 1], w), word(v[3][CH - 1], w), hf);
        }
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) {
          mma_bf16(o[nh][mt], a0, a1, a2, a3, bh[nh][0], bh[nh][1]);
          mma_bf16(o[nh][mt], a0, a1, a2, a3, bl[nh][0], bl[nh][1]);
        }
      }
    }
    fence_proxy_async_smem();  // this lane's reads of the stage before the copy that refills it
    __syncwarp();
    if (i + P::kStages < mine) issue(i + P::kStages);
  }

  // ---- merge the CTA's warps (the ring is free once every warp is here)
#pragma unroll
  for (int nh = 0; nh < NH; ++nh)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float l = lsum[nh][h];
      l += __shfl_xor_sync(kFull, l, 4);
      l += __shfl_xor_sync(kFull, l, 8);
      l += __shfl_xor_sync(kFull, l, 16);
      lsum[nh][h] = l;
    }
  __syncthreads();
  float* comb = reinterpret_cast<float*>(smem);  // [kWarps][16 heads][D]
  float* cm = comb + kWarps * 16 * D;            // [kWarps][16] max
  float* cl = cm + kWarps * 16;                  // [kWarps][16] sum
#pragma unroll
  for (int nh = 0; nh < NH; ++nh) {
    float* cw = comb + (warp * 16 + 8 * nh + 2 * qd) * D;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int d0 = D == 64 ? 8 * g + 2 * mt : 8 * g + mt;
      const int d1 = D == 64 ? d0 + 1 : d0 + 64;
      cw[d0] = o[nh][mt][0];
      cw[D + d0] = o[nh][mt][1];
      cw[d1] = o[nh][mt][2];
      cw[D + d1] = o[nh][mt][3];
    }
    if (g == 0) {
      cm[warp * 16 + 8 * nh + 2 * qd] = mrun[nh][0];
      cm[warp * 16 + 8 * nh + 2 * qd + 1] = mrun[nh][1];
      cl[warp * 16 + 8 * nh + 2 * qd] = lsum[nh][0];
      cl[warp * 16 + 8 * nh + 2 * qd + 1] = lsum[nh][1];
    }
  }
  __syncthreads();
  float* part = part0 + (size_t(j) * kGqaMaxSplits + s) * PS;
  for (int e = threadIdx.x; e < G * D; e += kThreads) {
    const int r = e / D, d = e - r * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, cm[w * 16 + r]);
    float O = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = exp2f(cm[w * 16 + r] - M);  // 0 for a warp without tiles
      O = fmaf(comb[(w * 16 + r) * D + d], f, O);
      L = fmaf(cl[w * 16 + r], f, L);
    }
    part[r * D + d] = O;
    if (d == 0) {
      part[G * D + r] = M;
      part[G * D + G + r] = L;
    }
  }
}

// One query head per CTA: o[h] = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s
// over the S split partials of its kv head, M = max_s m_s; thread
// (group sg, chunk c) sums splits sg, sg + NG, ... of dims 4c..4c+3 in
// order, then the groups are added in order: a fixed summation order.
template <int D>
__global__ void __launch_bounds__(kMergeThreads)
    gqa_merge_kernel(const float* __restrict__ part0, int G, int S, uint16_t* __restrict__ out) {
  constexpr int NC = D / 4;                // float4 chunks of a head
  constexpr int NG = kMergeThreads / NC;   // split groups
  __shared__ float wsh[kGqaMaxSplits];     // 2^(m_s - M) / L
  __shared__ float4 acc_sh[NG][NC];
  const int h = blockIdx.x, j = h / G, r = h - j * G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = tid % NC, sg = tid / NC;
  const int PS = partial_floats(G, D);
  const float* pj = part0 + size_t(j) * kGqaMaxSplits * PS;
  pdl_allow_next_grid();
  pdl_wait_prior_grid();  // the split kernel's partials
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 buf[kMergeBatch];
  auto load_batch = [&](int s0) {
#pragma unroll
    for (int b = 0; b < kMergeBatch; ++b) {
      const int s2 = s0 + NG * b;
      buf[b] = s2 < S ? __ldcg(reinterpret_cast<const float4*>(pj + size_t(s2) * PS + r * D + 4 * c))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  load_batch(sg);  // requested before the weights are known
  // warp 0: M = max m, L = sum l 2^(m - M), the weights 2^(m - M) / L
  if (warp == 0) {
    constexpr int kPer = kGqaMaxSplits / 32;
    float m[kPer], l[kPer];
    float M = -INFINITY;
#pragma unroll
    for (int b = 0; b < kPer; ++b) {
      const int s2 = lane + 32 * b;
      m[b] = s2 < S ? __ldcg(pj + size_t(s2) * PS + G * D + r) : -INFINITY;
      l[b] = s2 < S ? __ldcg(pj + size_t(s2) * PS + G * D + G + r) : 0.f;
      M = fmaxf(M, m[b]);
    }
    M = warp_max(M);
    float L = 0.f;
#pragma unroll
    for (int b = 0; b < kPer; ++b) {
      m[b] = lane + 32 * b < S ? exp2f(m[b] - M) : 0.f;
      L = fmaf(l[b], m[b], L);
    }
    const float inv = 1.f / warp_sum(L);
#pragma unroll
    for (int b = 0; b < kPer; ++b)
      if (lane + 32 * b < S) wsh[lane + 32 * b] = m[b] * inv;
  }
  __syncthreads();
  for (int s0 = sg;; s0 += NG * kMergeBatch) {
#pragma unroll
    for (int b = 0; b < kMergeBatch; ++b) {
      const int s2 = s0 + NG * b;
      const float w = s2 < S ? wsh[s2] : 0.f;
      acc.x = fmaf(buf[b].x, w, acc.x);
      acc.y = fmaf(buf[b].y, w, acc.y);
      acc.z = fmaf(buf[b].z, w, acc.z);
      acc.w = fmaf(buf[b].w, w, acc.w);
    }
    if (s0 + NG * kMergeBatch >= S) break;
    load_batch(s0 + NG * kMergeBatch);
  }
  acc_sh[sg][c] = acc;
  __syncthreads();
  if (sg == 0) {
#pragma unroll
    for (int g2 = 1; g2 < NG; ++g2) {
      const float4 a = acc_sh[g2][c];
      acc.x += a.x;
      acc.y += a.y;
      acc.z += a.z;
      acc.w += a.w;
    }
    const uint2 packed = make_uint2(
        uint32_t(f32_to_bf16_rne(acc.x)) | (uint32_t(f32_to_bf16_rne(acc.y)) << 16),
        uint32_t(f32_to_bf16_rne(acc.z)) | (uint32_t(f32_to_bf16_rne(acc.w)) << 16));
    *reinterpret_cast<uint2*>(out + int64_t(h) * D + 4 * c) = packed;
  }
}

// Tensor map over one cache: dims (head_dim, len, kv_heads), rows of
// head_dim bf16 at a stride of cap rows per kv head; box 64 x tok x 1, 128-byte
// swizzle; out-of-range rows (t >= len) read as zeros.
cudaError_t cache_map(CUtensorMap* map, const uint16_t* base, int D, int kv_heads, int64_t cap,
                      int64_t len, int tok) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(len), cuuint64_t(kv_heads)};
  const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(cap) * D * 2};
  const cuuint32_t box[3] = {64u, cuuint32_t(tok), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(base), dims, strides,
          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

template <int D, int NH>
cudaError_t launch_dn(const DeviceInfo& di, const uint16_t* q, const uint16_t* k,
                      const uint16_t* v, int G, int kv_heads, int64_t cap, int64_t len,
                      float scale, uint16_t* out, void* ws, cudaStream_t s, bool pdl) {
  using P = AttnPlan<D>;
  auto kern = gqa_decode_kernel<D, NH>;
  CUtensorMap tmk, tmv;
  if (cudaError_t e = cache_map(&tmk, k, D, kv_heads, cap, len, P::kTok)) return e;
  if (cudaError_t e = cache_map(&tmv, v, D, kv_heads, cap, len, P::kTok)) return e;
  if (cudaError_t e = ensure_smem(di, kern, P::kSmem)) return e;
  const int64_t T = (len + P::kTok - 1) / P::kTok;
  int64_t S = (di.sms + kv_heads - 1) / kv_heads;  // one CTA per SM over all kv heads
  if (S > T) S = T;
  if (S > kGqaMaxSplits) S = kGqaMaxSplits;
  if (S < 1) S = 1;
  const float sl2 = float(double(scale) * 1.4426950408889634);  // log2(e)
  float* part = static_cast<float*>(ws);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(S), unsigned(kv_heads));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = P::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmk, tmv, q, G, len, sl2, part,
                                         di.error_word))
    return e;
  // the merge always follows the split kernel programmatically
  cfg.gridDim = dim3(unsigned(G * kv_heads));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gqa_merge_kernel<D>, static_cast<const float*>(part), G,
                            int(S), out);
}

}  // namespace

size_t gqa_decode_workspace_bytes(int heads, int kv_heads, int head_dim) {
  const int G = heads / kv_heads;
  return size_t(kv_heads) * kGqaMaxSplits * size_t(partial_floats(G, head_dim)) * 4;
}

cudaError_t launch_gqa_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v, int heads,
                              int kv_heads, int head_dim, int64_t cap, int64_t len, float scale,
                              uint16_t* out, void* ws, cudaStream_t s, bool pdl) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorNoDevice;
  const int G = heads / kv_heads;
  if (head_dim == 64)
    return G > 8 ? launch_dn<64, 2>(*di, q, k, v, G, kv_heads, cap, len, scale, out, ws, s, pdl)
                 : launch_dn<64, 1>(*di, q, k, v, G, kv_heads, cap, len, scale, out, ws, s, pdl);
  if (head_dim == 128)
    return G > 8 ? launch_dn<128, 2>(*di, q, k, v, G, kv_heads, cap, len, scale, out, ws, s, pdl)
                 : launch_dn<128, 1>(*di, q, k, v, G, kv_heads, cap, len, scale, out, ws, s, pdl);
  return cudaErrorInvalidConfiguration;
}

}  // namespace tt
