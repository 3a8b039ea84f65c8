// quantize.cu -- MXFP8 quantizers (bf16 -> E4M3 payload + E8M0 scales),
// scale-factor packing for the attention kernels, and fused RMSNorm+Quantize.
//
// Format: OCP MX ("Low-Precision FlashAttention-4: End-to-End Block-Scaled
// Attention on Blackwell", section "Why MXFP8"): 32 elements share one
// power-of-two scale; the scale exponent is taken by bit extraction from the
// block maximum ("MXFP8 FlashAttention-4 Hits 2.85 Petaflops in Meta's
// Production Training", section "Inside the TMEM Bargain and Zero-Gather
// Jagged Pipeline").  Blocks run along the MMA K dimension: 1x32 along D for
// Q and K, 32x1 along tokens for V ("Meta's MXFP8 FlashAttention-4 kernel,
// tackling TMEM scale-factor constraints, hits up to 1.6x over BF16",
// paragraph 3), 32x32 squares for the backward operands (andresseo.expert,
// same section).  The fused producer follows brifing.si item 7.
//
// These kernels are HBM-bound: each thread owns an 8-column x 32-row slab in
// registers (16-byte loads, 8-byte stores, every byte read once).
#include <cuda_bf16.h>

#include "mx_ptx.cuh"
#include "mx_seq.cuh"
#include "mxfa_internal.h"

namespace mxfa {

static __device__ unsigned g_status_quant;

__device__ __forceinline__ uint4 ldg16(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// |bf16| bit patterns of a packed pair, as an unsigned max-able pair.
__device__ __forceinline__ uint32_t abs2(uint32_t w) { return w & 0x7FFF7FFFu; }
__device__ __forceinline__ uint32_t hmax2(uint32_t w) { return max(w & 0xFFFFu, w >> 16); }

// E8M0 from the bit pattern of a bf16 magnitude.
__device__ __forceinline__ uint32_t e8m0_from_bf16abs(uint32_t a) {
  if (a >= 0x7F80u) return 0xFFu;  // Inf or NaN in the block
  uint32_t e = a >> 7;
  return e > 8u ? e - 8u : 0u;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Eight bf16 (as uint4) times inv[0..7] -> eight E4M3 bytes (uint2).
__device__ __forceinline__ uint2 cvt8(uint4 v, const float* inv) {
  uint2 r;
  r.x = pack4_e4m3(bf_lo(v.x) * inv[0], bf_hi(v.x) * inv[1], bf_lo(v.y) * inv[2], bf_hi(v.y) * inv[3]);
  r.y = pack4_e4m3(bf_lo(v.z) * inv[4], bf_hi(v.z) * inv[5], bf_lo(v.w) * inv[6], bf_hi(v.w) * inv[7]);
  return r;
}

// ------------------------------------------------------------------ quantize
// grid (ceil(cols/1024), 4 * ceil(max_len/128), nseq), block 128.
// blockIdx.y indexes 32-row blocks of a sequence, including the padding blocks
// of its last 128-row tile (which only write padding scale bytes).
template <int MODE>
__global__ void __launch_bounds__(128) quant_kernel(QuantArgs a) {
  const int cols = a.H * a.D;
  const int col0 = blockIdx.x * 1024 + threadIdx.x * 8;
  const int g = blockIdx.z, rb = blockIdx.y;
  int64_t s0;
  int L;
  seq_info(a.seq, g, s0, L);
  const int nrb_real = (L + 31) / 32;
  const int nrb_pad = ((L + 127) / 128) * 4;
  if (rb >= nrb_pad || col0 >= cols) return;
  const int h = col0 / a.D, dcol = col0 % a.D;
  const int tile = rb >> 2, kb4 = rb & 3;
  int64_t tile_g = 0;
  if (a.sf_packed) tile_g = seq_units_before(a.seq, g, 128) + tile;
  if (a.sf_packed && tile_g >= a.packed_tiles) {
    atomicOr(&g_status_quant, DEV_BAD_INDEX);
    return;
  }
  const bool lead = (threadIdx.x & 3) == 0;  // first of the 4 threads of a 32-column block

  if (rb >= nrb_real) {  // padding rows of the last tile: scale bytes 0x7F only
    if (!a.sf_packed) return;
    if (MODE == 0) {
      uint8_t* base = a.sf_packed + (tile_g * a.H + h) * 512;
      if (lead)
        for (int r = 0; r < 32; r++) base[atom_off(kb4 * 32 + r, dcol / 32)] = 0x7F;
    } else if (MODE == 1) {
      uint8_t* base = a.sf_packed + (tile_g * a.H + h) * 512;
      for (int i = 0; i < 8; i++) base[atom_off(dcol + i, kb4)] = 0x7F;
    } else {
      if (lead) a.sf_packed[(tile_g * a.H + h) * 16 + kb4 * 4 + dcol / 32] = 0x7F;
    }
    return;
  }

  const int64_t r0 = s0 + int64_t(rb) * 32;
  const int nr = min(32, L - rb * 32);
  uint4 v[32];
#pragma unroll
  for (int r = 0; r < 32; r++)
    v[r] = r < nr ? ldg16(a.x + (r0 + r) * cols + col0) : make_uint4(0, 0, 0, 0);

  if (MODE == 0) {  // 1x32 along columns: 4 threads per block, per row
    const int ncb = cols / 32;
    uint8_t* pbase = a.sf_packed ? a.sf_packed + (tile_g * a.H + h) * 512 : nullptr;
#pragma unroll
    for (int r = 0; r < 32; r++) {
      uint32_t m = max(max(hmax2(abs2(v[r].x)), hmax2(abs2(v[r].y))),
                       max(hmax2(abs2(v[r].z)), hmax2(abs2(v[r].w))));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      if (r < nr) {
        uint32_t s = e8m0_from_bf16abs(m);
        uint2 out;
        if (s == 0xFFu) {
          out = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
        } else {
          float inv[8];
          float f = e8m0_inv_scale(s);
#pragma unroll
          for (int i = 0; i < 8; i++) inv[i] = f;
          out = cvt8(v[r], inv);
        }
        *reinterpret_cast<uint2*>(a.data + (r0 + r) * cols + col0) = out;
        if (lead) {
          if (a.sf_compact) a.sf_compact[(r0 + r) * ncb + col0 / 32] = uint8_t(s);
          if (pbase) pbase[atom_off(kb4 * 32 + r, dcol / 32)] = uint8_t(s);
        }
      } else if (lead && pbase) {
        pbase[atom_off(kb4 * 32 + r, dcol / 32)] = 0x7F;
      }
    }
  } else {
    // per-column maxima over the 32 rows (pairs of columns per word)
    uint32_t cm[4] = {0, 0, 0, 0};
#pragma unroll
    for (int r = 0; r < 32; r++) {
      cm[0] = __vmaxu2(cm[0], abs2(v[r].x));
      cm[1] = __vmaxu2(cm[1], abs2(v[r].y));
      cm[2] = __vmaxu2(cm[2], abs2(v[r].z));
      cm[3] = __vmaxu2(cm[3], abs2(v[r].w));
    }
    const int64_t b32 = seq_units_before(a.seq, g, 32) + rb;
    uint32_t s[8];
    float inv[8];
    if (MODE == 1) {
#pragma unroll
      for (int i = 0; i < 4; i++) {
        s[2 * i] = e8m0_from_bf16abs(cm[i] & 0xFFFFu);
        s[2 * i + 1] = e8m0_from_bf16abs(cm[i] >> 16);
      }
    } else {
      uint32_t m = max(max(hmax2(cm[0]), hmax2(cm[1])), max(hmax2(cm[2]), hmax2(cm[3])));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      uint32_t sb = e8m0_from_bf16abs(m);
#pragma unroll
      for (int i = 0; i < 8; i++) s[i] = sb;
    }
    bool bad[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
      bad[i] = s[i] == 0xFFu;
      inv[i] = bad[i] ? 0.0f : e8m0_inv_scale(s[i]);
    }
#pragma unroll
    for (int r = 0; r < 32; r++) {
      if (r < nr) {
        uint2 out = cvt8(v[r], inv);
        uint8_t* ob = reinterpret_cast<uint8_t*>(&out);
#pragma unroll
        for (int i = 0; i < 8; i++)
          if (bad[i]) ob[i] = 0x7F;
        *reinterpret_cast<uint2*>(a.data + (r0 + r) * cols + col0) = out;
      }
    }
    if (MODE == 1) {
      if (a.sf_compact) {
        uint2 sv;
        sv.x = s[0] | (s[1] << 8) | (s[2] << 16) | (s[3] << 24);
        sv.y = s[4] | (s[5] << 8) | (s[6] << 16) | (s[7] << 24);
        *reinterpret_cast<uint2*>(a.sf_compact + b32 * cols + col0) = sv;
      }
      if (a.sf_packed) {
        uint8_t* base = a.sf_packed + (tile_g * a.H + h) * 512;
#pragma unroll
        for (int i = 0; i < 8; i++) base[atom_off(dcol + i, kb4)] = uint8_t(s[i]);
      }
    } else if (lead) {
      if (a.sf_compact) a.sf_compact[b32 * (cols / 32) + col0 / 32] = uint8_t(s[0]);
      if (a.sf_packed) a.sf_packed[(tile_g * a.H + h) * 16 + kb4 * 4 + dcol / 32] = uint8_t(s[0]);
    }
  }
}

cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t st) {
  const int cols = a.H * a.D;
  dim3 grid((cols + 1023) / 1024, 4 * ((a.seq.seqlen + 127) / 128), a.seq.nseq);
  if (grid.y == 0 || grid.z == 0) return cudaSuccess;
  switch (a.mode) {
    case 0: quant_kernel<0><<<grid, 128, 0, st>>>(a); break;
    case 1: quant_kernel<1><<<grid, 128, 0, st>>>(a); break;
    default: quant_kernel<2><<<grid, 128, 0, st>>>(a); break;
  }
  return cudaPeekAtLastError();
}

// ------------------------------------------------------------------ sf pack
// Compact scales -> packed (MMA atom) scales, values unchanged; padding 0x7F.
// grid (4 * ceil(max_len/128), nseq), block 256.
__global__ void __launch_bounds__(256) sf_pack_kernel(PackArgs a) {
  const int cols = a.H * a.D;
  const int ncb = cols / 32;
  const int g = blockIdx.y, rb = blockIdx.x;
  int64_t s0;
  int L;
  seq_info(a.seq, g, s0, L);
  const int nrb_real = (L + 31) / 32;
  if (rb >= ((L + 127) / 128) * 4) return;
  const int tile = rb >> 2, kb4 = rb & 3;
  const int64_t tile_g = seq_units_before(a.seq, g, 128) + tile;
  if (tile_g >= a.packed_tiles) {
    atomicOr(&g_status_quant, DEV_BAD_INDEX);
    return;
  }
  const bool real = rb < nrb_real;
  if (a.mode == 0) {
    for (int i = threadIdx.x; i < 32 * ncb; i += blockDim.x) {
      int r = i / ncb, cb = i % ncb;
      int h = cb / (a.D / 32), kb = cb % (a.D / 32);
      bool valid = real && rb * 32 + r < L;
      uint8_t v = valid ? a.sf_compact[(s0 + rb * 32 + r) * ncb + cb] : 0x7F;
      a.sf_packed[(tile_g * a.H + h) * 512 + atom_off(kb4 * 32 + r, kb)] = v;
    }
  } else {
    const int64_t b32 = seq_units_before(a.seq, g, 32) + rb;
    if (a.mode == 1) {
      for (int c = threadIdx.x; c < cols; c += blockDim.x) {
        int h = c / a.D, d = c % a.D;
        uint8_t v = real ? a.sf_compact[b32 * cols + c] : 0x7F;
        a.sf_packed[(tile_g * a.H + h) * 512 + atom_off(d, kb4)] = v;
      }
    } else {
      for (int cb = threadIdx.x; cb < ncb; cb += blockDim.x) {
        int h = cb / (a.D / 32), kb = cb % (a.D / 32);
        uint8_t v = real ? a.sf_compact[b32 * ncb + cb] : 0x7F;
        a.sf_packed[(tile_g * a.H + h) * 16 + kb4 * 4 + kb] = v;
      }
    }
  }
}

cudaError_t launch_sf_pack(const PackArgs& a, cudaStream_t st) {
  dim3 grid(4 * ((a.seq.seqlen + 127) / 128), a.seq.nseq);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  sf_pack_kernel<<<grid, 256, 0, st>>>(a);
  return cudaPeekAtLastError();
}

// ---------------------------------------------------------- RMSNorm+Quantize
// One CTA = 32 rows, warp w = row w; lane l owns columns 8l + 256k + j.
// Sum of squares in that order (k outer, j inner), then a butterfly over
// 16, 8, 4, 2, 1; mean = ss / C; r = 1 / sqrt(mean + eps); y = (x * r) * gamma,
// each a correctly rounded fp32 operation.  Column (32x1) and square (32x32)
// maxima are exchanged through shared memory, one 256-column chunk at a time.
template <int NK>
__global__ void __launch_bounds__(1024, 1) rms_quant_kernel(RmsArgs a) {
  __shared__ uint32_t sm_abs[32][257];
  __shared__ uint32_t sm_part[4][256];
  __shared__ float sm_colinv[256];
  __shared__ float sm_sqinv[8];
  __shared__ uint8_t sm_colbad[256];
  constexpr int C = NK * 256;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, t = threadIdx.x;
  const int64_t row = int64_t(blockIdx.x) * 32 + w;
  const bool valid = row < a.T;
  const bool want_cs = a.col_data || a.sq_data;
  const int64_t seg = row / a.seg_len;       // sequence of this row (packed layouts)
  const int64_t pos = row % a.seg_len;       // position in the sequence
  const int64_t tiles_per_seq = a.seg_len / 128;
  const int64_t tile_g = seg * tiles_per_seq + pos / 128;
  const int rr = int(pos % 128);
  const int kb4 = int(pos % 128) / 32;  // same for all rows of the CTA (seg_len % 32 == 0)

  uint4 xv[NK];
#pragma unroll
  for (int k = 0; k < NK; k++)
    xv[k] = valid ? ldg16(a.x + row * C + 256 * k + 8 * l) : make_uint4(0, 0, 0, 0);

  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < NK; k++) {
    const uint32_t wv[4] = {xv[k].x, xv[k].y, xv[k].z, xv[k].w};
#pragma unroll
    for (int j = 0; j < 4; j++) {
      float lo = bf_lo(wv[j]), hi = bf_hi(wv[j]);
      ss = __fadd_rn(ss, __fmul_rn(lo, lo));
      ss = __fadd_rn(ss, __fmul_rn(hi, hi));
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, off));
  const float mean = __fdiv_rn(ss, float(C));
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, a.eps)));

#pragma unroll
  for (int k = 0; k < NK; k++) {
    const int c0 = 256 * k + 8 * l;
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(a.gamma + c0));
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(a.gamma + c0 + 4));
    const float gm[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const uint32_t wv[4] = {xv[k].x, xv[k].y, xv[k].z, xv[k].w};
    float y[8];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      y[2 * j] = __fmul_rn(__fmul_rn(bf_lo(wv[j]), r), gm[2 * j]);
      y[2 * j + 1] = __fmul_rn(__fmul_rn(bf_hi(wv[j]), r), gm[2 * j + 1]);
    }
    uint32_t am = 0;
#pragma unroll
    for (int j = 0; j < 8; j++) am = max(am, __float_as_uint(y[j]) & 0x7FFFFFFFu);
    const int h = c0 / a.D, d0 = c0 % a.D;

    if (a.row_data) {  // 1x32 along C: 4 lanes per block
      uint32_t m = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      uint32_t s = m >= 0x7F800000u ? 0xFFu : e8m0_from_amax(__uint_as_float(m));
      float f = s == 0xFFu ? 0.0f : e8m0_inv_scale(s);
      uint2 out;
      out.x = pack4_e4m3(y[0] * f, y[1] * f, y[2] * f, y[3] * f);
      out.y = pack4_e4m3(y[4] * f, y[5] * f, y[6] * f, y[7] * f);
      if (s == 0xFFu) out = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
      if (valid) {
        *reinterpret_cast<uint2*>(a.row_data + row * C + c0) = out;
        if ((l & 3) == 0) {
          if (a.row_sfc) a.row_sfc[row * (C / 32) + c0 / 32] = uint8_t(s);
          if (a.row_sfp) a.row_sfp[(tile_g * a.H + h) * 512 + atom_off(rr, d0 / 32)] = uint8_t(s);
        }
      }
    }
    if (want_cs) {
#pragma unroll
      for (int j = 0; j < 8; j++) sm_abs[w][8 * l + j] = __float_as_uint(y[j]) & 0x7FFFFFFFu;
      __syncthreads();
      {
        const int c = t & 255, part = t >> 8;
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) m = max(m, sm_abs[part * 8 + i][c]);
        sm_part[part][c] = m;
      }
      __syncthreads();
      if (t < 256) {
        uint32_t m = max(max(sm_part[0][t], sm_part[1][t]), max(sm_part[2][t], sm_part[3][t]));
        const int cc = 256 * k + t, hh = cc / a.D, dd = cc % a.D;
        uint32_t s = m >= 0x7F800000u ? 0xFFu : e8m0_from_amax(__uint_as_float(m));
        sm_colinv[t] = s == 0xFFu ? 0.0f : e8m0_inv_scale(s);
        sm_colbad[t] = s == 0xFFu;
        if (a.col_data) {
          if (a.col_sfc) a.col_sfc[int64_t(blockIdx.x) * C + cc] = uint8_t(s);
          if (a.col_sfp) a.col_sfp[(tile_g * a.H + hh) * 512 + atom_off(dd, kb4)] = uint8_t(s);
        }
        // one warp = 32 columns = one square block
        uint32_t bm = m;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) bm = max(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, off));
        if (l == 0) {
          uint32_t sq = bm >= 0x7F800000u ? 0xFFu : e8m0_from_amax(__uint_as_float(bm));
          sm_sqinv[w] = sq == 0xFFu ? -1.0f : e8m0_inv_scale(sq);
          if (a.sq_data) {
            if (a.sq_sfc) a.sq_sfc[int64_t(blockIdx.x) * (C / 32) + 8 * k + w] = uint8_t(sq);
            if (a.sq_sfp) a.sq_sfp[(tile_g * a.H + hh) * 16 + kb4 * 4 + dd / 32] = uint8_t(sq);
          }
        }
      }
      __syncthreads();
      if (valid && a.col_data) {
        uint2 out;
        const float* ci = sm_colinv + 8 * l;
        out.x = pack4_e4m3(y[0] * ci[0], y[1] * ci[1], y[2] * ci[2], y[3] * ci[3]);
        out.y = pack4_e4m3(y[4] * ci[4], y[5] * ci[5], y[6] * ci[6], y[7] * ci[7]);
        uint8_t* ob = reinterpret_cast<uint8_t*>(&out);
#pragma unroll
        for (int j = 0; j < 8; j++)
          if (sm_colbad[8 * l + j]) ob[j] = 0x7F;
        *reinterpret_cast<uint2*>(a.col_data + row * C + c0) = out;
      }
      if (valid && a.sq_data) {
        const float f = sm_sqinv[l >> 2];
        uint2 out;
        if (f < 0.0f) {
          out = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
        } else {
          out.x = pack4_e4m3(y[0] * f, y[1] * f, y[2] * f, y[3] * f);
          out.y = pack4_e4m3(y[4] * f, y[5] * f, y[6] * f, y[7] * f);
        }
        *reinterpret_cast<uint2*>(a.sq_data + row * C + c0) = out;
      }
      __syncthreads();
    }
  }
}

cudaError_t launch_rmsnorm_quant(const RmsArgs& a, cudaStream_t st) {
  dim3 grid(unsigned((a.T + 31) / 32));
  if (grid.x == 0) return cudaSuccess;
  switch (a.C) {
    case 256: rms_quant_kernel<1><<<grid, 1024, 0, st>>>(a); break;
    case 512: rms_quant_kernel<2><<<grid, 1024, 0, st>>>(a); break;
    case 1024: rms_quant_kernel<4><<<grid, 1024, 0, st>>>(a); break;
    case 2048: rms_quant_kernel<8><<<grid, 1024, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaPeekAtLastError();
}

unsigned read_status_quant(cudaStream_t st) {
  unsigned v = 0, z = 0;
  cudaMemcpyFromSymbolAsync(&v, g_status_quant, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
  cudaMemcpyToSymbolAsync(g_status_quant, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
  cudaStreamSynchronize(st);
  return v;
}

}  // namespace mxfa
