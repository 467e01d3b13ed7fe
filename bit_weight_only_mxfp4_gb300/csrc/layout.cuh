// Packed device layouts shared by the loader kernels and the matvec kernels.
#pragma once

#include <cstdint>

namespace tt {

// Packed gate/up ("swiglu") layout: one record per output row r, records
// back to back:
//
//   [gate codes  k/2 B][up codes  k/2 B][gate scales k/32 B][up scales k/32 B]
//   [pad to 8][post_g f32][post_u f32][pad to 16]
//
// so one bulk copy brings everything a row pair needs (codes, scales and
// both postscales) into shared memory, and every code chunk sits at a
// 16-byte offset.  Codes and scales keep the canonical bytes unchanged.
struct SwigluRecord {
  int k;     // reduction length (multiple of 32)
  int nblk;  // k / 32
  int post;  // byte offset of post_g (post_u follows)
  int bytes; // record size, multiple of 16

  __host__ __device__ explicit SwigluRecord(int k_) : k(k_), nblk(k_ >> 5) {
    post = (k + 2 * nblk + 7) & ~7;
    bytes = (post + 8 + 15) & ~15;
  }
  __host__ __device__ int gate_codes() const { return 0; }
  __host__ __device__ int up_codes() const { return k >> 1; }
  __host__ __device__ int gate_scales() const { return k; }
  __host__ __device__ int up_scales() const { return k + nblk; }
};

// Packed single-matrix layout used for the MoE down projections, sliced by
// COLUMNS so that a CTA owning a 16-wide slice of the reduction index (the
// experts' SwiGLU outputs it computed itself) reads that slice of every row
// as one contiguous run:
//
//   codes : [k/16 slices][n rows][8 B]   (the row's canonical code bytes
//                                         8s .. 8s+7, i.e. k = 16s .. 16s+15)
//   scales: [k/32 blocks][n rows][1 B]   (the row's E8M0 byte of block b)
//
// each region padded to 16 bytes.  Codes and scales keep their bytes.
struct ColSlices {
  int64_t n;
  int k, nslice, nblk;
  int64_t codes_bytes, scales_off, bytes;
  __host__ __device__ ColSlices(int64_t n_, int k_) : n(n_), k(k_), nslice(k_ >> 4), nblk(k_ >> 5) {
    codes_bytes = (n * (k >> 1) + 15) & ~int64_t(15);
    scales_off = codes_bytes;
    bytes = scales_off + ((n * nblk + 15) & ~int64_t(15));
  }
  // byte offset of (slice s, row r)'s 8 code bytes / of (block b, row r)'s scale
  __host__ __device__ int64_t code_at(int s, int64_t r) const { return ((int64_t)s * n + r) * 8; }
  __host__ __device__ int64_t scale_at(int b, int64_t r) const {
    return scales_off + (int64_t)b * n + r;
  }
};

}  // namespace tt
