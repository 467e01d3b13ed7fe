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

// Packed single-matrix ("rows") layout used for the MoE down projection:
//   [codes k/2 B][scales k/32 B][pad to 16]
struct RowRecord {
  int k, nblk, bytes;
  __host__ __device__ explicit RowRecord(int k_) : k(k_), nblk(k_ >> 5) {
    bytes = (k / 2 + nblk + 15) & ~15;
  }
  __host__ __device__ int codes() const { return 0; }
  __host__ __device__ int scales() const { return k >> 1; }
};

}  // namespace tt
