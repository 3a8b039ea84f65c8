// mx_seq.cuh -- sequence geometry helpers shared by the kernels: where a
// sequence starts, its length, and the offsets of its rows in the compact
// (32-row block) and packed (128-row tile) scale-factor layouts.
#pragma once
#include "mxfa_internal.h"

namespace mxfa {

__device__ __forceinline__ void seq_info(const Seqs& s, int g, int64_t& start, int& len) {
  if (s.cu) {
    int a = __ldg(s.cu + g), b = __ldg(s.cu + g + 1);
    start = a;
    len = b - a;
  } else {
    start = int64_t(g) * s.seqlen;
    len = s.seqlen;
  }
}

// Sum over sequences i < g of ceil(len_i / gran).
__device__ __forceinline__ int64_t seq_units_before(const Seqs& s, int g, int gran) {
  if (!s.cu) return int64_t(g) * ((s.seqlen + gran - 1) / gran);
  int64_t acc = 0;
  int prev = __ldg(s.cu);
#pragma unroll 8
  for (int i = 0; i < g; i++) {
    int nx = __ldg(s.cu + i + 1);
    acc += (nx - prev + gran - 1) / gran;
    prev = nx;
  }
  return acc;
}

// seq_units_before computed by a whole (converged) warp: lane l sums the
// sequences l, l + 32, ... and a butterfly adds the lanes' sums.  Every lane
// returns the total.
__device__ __forceinline__ int64_t seq_units_before_warp(const Seqs& s, int g, int gran, int lane) {
  if (!s.cu) return int64_t(g) * ((s.seqlen + gran - 1) / gran);
  long long acc = 0;
  for (int i = lane; i < g; i += 32) acc += (__ldg(s.cu + i + 1) - __ldg(s.cu + i) + gran - 1) / gran;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  return acc;
}

// Byte offset of (row r in tile, k-block kb) inside a 512-byte MMA scale atom:
// 128 rows x 4 k-blocks, rows split as (r % 32, r / 32).
__host__ __device__ __forceinline__ int atom_off(int r, int kb) {
  return (r & 31) * 16 + (r >> 5) * 4 + kb;
}

}  // namespace mxfa
