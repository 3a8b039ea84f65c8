// gemm.cu -- MXFP8 projection GEMM with a quantizing epilogue, for sm_103a.
//
// What it computes ("MXFP8 FlashAttention-4 Hits 2.85 Petaflops in Meta's
// Production Training", section "Inside the TMEM Bargain and Zero-Gather
// Jagged Pipeline": quantization fused into the projection GEMM's epilogue;
// "Meta's FlashAttention-4 Achieves 2.85 PF/s with MXFP8 on Blackwell GPUs",
// item 7: GEMM+Quantize emitting FP8 with dual scale-factor layouts):
//   Y = A B^T with A [M][K] and B [N][K] MXFP8 (E4M3, E8M0 scale per 32
//   along K) -- or MXFP6 / MXFP4 operands (runs of 16 codes packed and padded
//   to 16 bytes, one byte per element), which the same MMA kind reads (the
//   pages' next formats) -- fp32 accumulation in tensor
//   memory, and an epilogue that writes
//   Y as bf16 and/or as MXFP8 in two block layouts -- 1x32 along N (ROW: the
//   next GEMM's K dimension, e.g. Q and K of attention) and 32x1 along M
//   (COL: e.g. V of attention, whose MMA K dimension is the token axis) --
//   with compact and packed scales, one pass over the accumulator.
//
// Structure: persistent, one CTA per SM, 128x128 output tiles (N tiles
// fastest, so that a wave of CTAs reads few A panels and B stays in L2), 6 warps:
//   warp 0      TMA producer: per 128-wide K step, the A and B tiles (128 x
//               128 E4M3, 128B swizzle) and their 512-byte scale atoms into a
//               6-stage ring
//   warp 1      TMEM owner and MMA issuer: scale atoms into TMEM by
//               tcgen05.cp, four block-scaled MMAs (K = 32 each) per stage;
//               two accumulators, so one tile's epilogue overlaps the next
//               tile's MMAs
//   warps 2-    epilogue, EQ warps per TMEM lane quadrant (128 / EQ columns each):
//               thread = output row = TMEM lane; each 32-column
//               chunk is one ROW block of the thread, and 32 rows of a warp
//               form the COL blocks (block maximum by a warp reduction)
// TMEM: accumulators [0,128) and [128,256); per stage s the A / B scale
// slots at 256 + 8s and 256 + 8s + 4.
#include <cuda_bf16.h>

#include "mx_ptx.cuh"
#include "mx_seq.cuh"
#include "mxfa_internal.h"

namespace mxfa {

static __device__ unsigned g_status_gemm;

namespace gemm {
constexpr int BM = 128, BN = 128, BK = 128;
constexpr int NS = 6;
constexpr int TILE_BYTES = 128 * 128;
constexpr int STAGE_BYTES = 2 * TILE_BYTES + 1024;  // A, B, A atom, B atom
constexpr int OFF_BAR = NS * STAGE_BYTES;
enum { B_FULL = 0, B_EMPTY = B_FULL + NS, B_ACCFULL = B_EMPTY + NS, B_ACCEMPTY = B_ACCFULL + 2, B_TEAR = B_ACCEMPTY + 2, NBAR };
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "GEMM stages exceed the shared memory of one CTA");
constexpr uint32_t COL_ACC = 0, COL_SF = 256;
#ifndef MXFA_GEMM_EQ
#define MXFA_GEMM_EQ 2
#endif
constexpr int EQ = MXFA_GEMM_EQ;            // epilogue warps per TMEM lane quadrant
constexpr int CPW = 4 / EQ;                 // 32-column chunks per epilogue warp
constexpr int NTHREADS = 64 + 128 * EQ;     // producer, MMA issuer, 4 EQ epilogue warps
}  // namespace gemm

__device__ __forceinline__ bool gemm_wait_raw(uint32_t bar, uint32_t parity) {
  unsigned long long t0 = global_ns();
  while (!mbar_try_wait_sleep(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

// Largest |x| bit pattern over the 32 lanes (non-negative floats order like
// their bit patterns; Inf and NaN compare above every finite value).
__device__ __forceinline__ uint32_t warp_max_abs_bits(float x) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(__float_as_uint(x) & 0x7FFFFFFFu));
  return r;
}

// Largest |x| of a, b, c, NaN if any of them is NaN (Inf stays Inf).
__device__ __forceinline__ float max3_abs_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(fabsf(a)), "f"(fabsf(b)), "f"(fabsf(c)));
  return r;
}
// 32 fp32 values times one inverse scale f -> 32 E4M3 bytes at dst (16-byte
// aligned); bad (a 0xFF scale: Inf / NaN in the block) gives 0x7F bytes.
__device__ __forceinline__ void store_e4m3_32_uniform(uint8_t* dst, const float* y, float f, bool bad) {
  uint32_t w[8];
  const float2 f2 = make_float2(f, f);
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const float2 a = fmul2(make_float2(y[4 * i], y[4 * i + 1]), f2);
    const float2 b = fmul2(make_float2(y[4 * i + 2], y[4 * i + 3]), f2);
    w[i] = bad ? 0x7F7F7F7Fu : (cvt_e4m3x2(a.x, a.y) | (cvt_e4m3x2(b.x, b.y) << 16));
  }
  reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
  reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// 32 fp32 values -> 32 E4M3 bytes at dst (16-byte aligned), each value times
// its own inverse scale inv[i]; a 0xFF scale (Inf / NaN in the block) gives 0x7F.
__device__ __forceinline__ void store_e4m3_32(uint8_t* dst, const float* y, const float* inv, const uint32_t* sc) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; i++) {
    uint32_t lo = cvt_e4m3x2(y[4 * i] * inv[4 * i], y[4 * i + 1] * inv[4 * i + 1]);
    uint32_t hi = cvt_e4m3x2(y[4 * i + 2] * inv[4 * i + 2], y[4 * i + 3] * inv[4 * i + 3]);
    if (sc[4 * i] == 0xFFu) lo = (lo & 0xFF00u) | 0x7Fu;
    if (sc[4 * i + 1] == 0xFFu) lo = (lo & 0x00FFu) | 0x7F00u;
    if (sc[4 * i + 2] == 0xFFu) hi = (hi & 0xFF00u) | 0x7Fu;
    if (sc[4 * i + 3] == 0xFFu) hi = (hi & 0x00FFu) | 0x7F00u;
    w[i] = lo | (hi << 16);
  }
  reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
  reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

__global__ void __launch_bounds__(gemm::NTHREADS, 1) gemm_quant_kernel(const __grid_constant__ GemmArgs a) {
  using namespace gemm;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt_n = int(a.M / BM), nt_n = int(a.N / BN), kt_n = int(a.K / BK);
  const int ntiles = mt_n * nt_n;

  const uint32_t bar0 = base + OFF_BAR;
  auto BAR = [&](int i) { return bar0 + 8u * uint32_t(i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 8);
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < NS; s++) {
      mbar_init(BAR(B_FULL + s), 1);
      mbar_init(BAR(B_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(BAR(B_ACCFULL + b), 1);
      mbar_init(BAR(B_ACCEMPTY + b), 4 * EQ);  // one arrival per epilogue warp
    }
    mbar_init(BAR(B_TEAR), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&a.tm_a);
      tma_prefetch_desc(&a.tm_b);
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
        const int mt = t / nt_n, nt = t % nt_n;  // N tiles fastest: a wave shares few A panels, B stays in L2
        for (int kk = 0; kk < kt_n; kk++, it++) {
          const int s = it % NS;
          if (it >= NS && !mbar_wait(BAR(B_EMPTY + s), ((it / NS) - 1) & 1, abort_flag, &g_status_gemm)) {
            ok = false;
            break;
          }
          const uint32_t st = base + s * STAGE_BYTES;
          const uint32_t fb = BAR(B_FULL + s);
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          tma_load_3d(st, &a.tm_a, fb, 0, kk, mt * BM);
          tma_load_3d(st + TILE_BYTES, &a.tm_b, fb, 0, kk, nt * BN);
          bulk_load(st + 2 * TILE_BYTES, a.sfa + (int64_t(mt) * kt_n + kk) * 512, 512, fb);
          bulk_load(st + 2 * TILE_BYTES + 512, a.sfb + (int64_t(nt) * kt_n + kk) * 512, 512, fb);
        }
      }
      // every issued copy has landed before the CTA may exit
      for (int j = max(0, it - NS); j < it; j++) gemm_wait_raw(BAR(B_FULL + j % NS), (j / NS) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t tm = __shfl_sync(0xFFFFFFFFu, tmem, 0);
    auto wait_all = [&](uint32_t bar, uint32_t par) {
      return __all_sync(0xFFFFFFFFu, mbar_wait(bar, par, abort_flag, &g_status_gemm));
    };
    int it = 0, lt = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x, lt++) {
      const int b = lt & 1;
      // accumulator b was drained by the epilogue (use lt / 2 - 1)
      if (lt >= 2 && !wait_all(BAR(B_ACCEMPTY + b), ((lt >> 1) - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kk = 0; kk < kt_n; kk++, it++) {
        const int s = it % NS;
        if (!wait_all(BAR(B_FULL + s), (it / NS) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = base + s * STAGE_BYTES;
        const uint32_t sfa = COL_SF + 8u * s, sfb = sfa + 4;
        tc_cp_sf_w(tm + sfa, smem_desc(st + 2 * TILE_BYTES, 128, 128, 0));
        tc_cp_sf_w(tm + sfb, smem_desc(st + 2 * TILE_BYTES + 512, 128, 128, 0));
        const uint64_t dA = smem_desc(st, 16, 1024, 2);
        const uint64_t dB = smem_desc(st + TILE_BYTES, 16, 1024, 2);
#pragma unroll
        for (int k = 0; k < 4; k++)
          mma_mxf8_ss_w(tm + COL_ACC + 128u * b, dA + uint64_t(2 * k), dB + uint64_t(2 * k),
                        idesc_mxf8(128, 128, 0, 0, k, k, a.a_fmt, a.b_fmt), tm + sfa, tm + sfb,
                        (kk > 0 || k > 0) ? 1u : 0u);
        tc_commit_w(BAR(B_EMPTY + s));  // the stage (and its scale slots) may be refilled
      }
      if (ok) tc_commit_w(BAR(B_ACCFULL + b));
    }
    tc_commit_w(BAR(B_TEAR));
    gemm_wait_raw(BAR(B_TEAR), 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // EQ warps per TMEM lane quadrant, each taking CPW 32-column chunks of the
    // tile's 128 columns for the quadrant's 32 rows.
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int part = (warp - 2) >> 2;       // columns [32 CPW part, 32 CPW (part + 1))
    const int r = q * 32 + lane;            // row of the tile
    const uint32_t lane_base = uint32_t(q * 32) << 16;
    int lt = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, lt++) {
      const int b = lt & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(BAR(B_ACCFULL + b), (lt >> 1) & 1, abort_flag, &g_status_gemm)))
        break;
      tc_fence_after();
      float y[32 * CPW];
#pragma unroll
      for (int c = 0; c < CPW; c++)
        tmem_ld32(tmem + lane_base + COL_ACC + 128u * b + 32u * (CPW * part + c),
                  reinterpret_cast<uint32_t*>(y) + 32 * c);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < CPW; c++) reg_fence32(reinterpret_cast<uint32_t*>(y) + 32 * c);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_ACCEMPTY + b));  // the MMAs may reuse accumulator b
      const int mt = t / nt_n, nt = t % nt_n;  // N tiles fastest: a wave shares few A panels, B stays in L2
      const int64_t m = int64_t(mt) * BM + r;
      uint32_t row_sc = 0;  // this warp's CPW ROW scale bytes
#pragma unroll
      for (int c = 0; c < CPW; c++) {
        const float* yc = y + 32 * c;
        const int cg = CPW * part + c;  // 32-column chunk of the tile
        const int64_t n0 = int64_t(nt) * BN + 32 * cg;
        if (a.y_bf16) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; e++) {
            __nv_bfloat162 p2 = __floats2bfloat162_rn(yc[2 * e], yc[2 * e + 1]);
            w[e] = *reinterpret_cast<uint32_t*>(&p2);
          }
          uint4* dst = reinterpret_cast<uint4*>(a.y_bf16 + m * a.N + n0);
#pragma unroll
          for (int v4 = 0; v4 < 4; v4++) dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
        }
        if (a.row_data) {
          // ROW: this thread's 32 values are one 1x32 block along N; the
          // NaN-propagating maximum also flags Inf / NaN (exponent field 0xFF)
          float mx = max3_abs_nan(yc[0], yc[1], yc[2]);
#pragma unroll
          for (int i = 3; i < 31; i += 2) mx = max3_abs_nan(mx, yc[i], yc[i + 1]);
          mx = max3_abs_nan(mx, yc[31], 0.0f);
          const uint32_t sc = e8m0_from_amax(mx);
          row_sc |= sc << (8 * c);
          store_e4m3_32_uniform(a.row_data + m * a.N + n0, yc, sc == 0xFFu ? 1.0f : e8m0_inv_scale(sc), sc == 0xFFu);
        }
        if (a.col_data) {
          // COL: the warp's 32 rows form one 32x1 block per column
          float inv[32];
          uint32_t scs[32];
          uint32_t my_sc = 0;
#pragma unroll
          for (int i = 0; i < 32; i++) {
            const uint32_t mb = warp_max_abs_bits(yc[i]);
            const uint32_t e = mb >> 23;
            const uint32_t sc = e == 0xFFu ? 0xFFu : (e > 8u ? e - 8u : 0u);
            scs[i] = sc;
            inv[i] = sc == 0xFFu ? 1.0f : e8m0_inv_scale(sc);
            if (i == lane) my_sc = sc;
          }
          store_e4m3_32(a.col_data + m * a.N + n0, yc, inv, scs);
          const int64_t rb = int64_t(mt) * 4 + q;  // 32-row block
          if (a.col_sfc) a.col_sfc[rb * a.N + n0 + lane] = uint8_t(my_sc);
          // packed COL atom of (row tile mt, column group nt): byte (d % 32) * 16 + (d / 32) * 4 + k
          if (a.col_sfp)
            a.col_sfp[(int64_t(mt) * nt_n + nt) * 512 + atom_off(32 * cg + lane, q)] = uint8_t(my_sc);
        }
      }
      if (a.row_data) {
#pragma unroll
        for (int c = 0; c < CPW; c++) {
          const uint8_t v = uint8_t(row_sc >> (8 * c));
          if (a.row_sfc) a.row_sfc[m * (a.N / 32) + int64_t(nt) * 4 + CPW * part + c] = v;
          if (a.row_sfp)
            a.row_sfp[(int64_t(mt) * nt_n + nt) * 512 + (r & 31) * 16 + (r >> 5) * 4 + CPW * part + c] = v;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_gemm_quant(const GemmArgs& a, cudaStream_t st) {
  static std::atomic<unsigned long long> attr{0};
  clear_stale_error();
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(gemm_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                gemm::SMEM_BYTES);
  });
  if (e != cudaSuccess) return e;
  const int64_t ntiles = (a.M / gemm::BM) * (a.N / gemm::BN);
  if (ntiles == 0 || a.K == 0) return cudaSuccess;
  const int sms = sm_count_current_device();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const unsigned grid = unsigned(ntiles < sms ? ntiles : sms);
  gemm_quant_kernel<<<grid, gemm::NTHREADS, gemm::SMEM_BYTES, st>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------ peak probe
// Back-to-back block-scaled MMAs (M = 128, N = 256, K = 32 E4M3) on operands
// resident in shared memory, one CTA per SM: the tensor pipe's own peak on
// this GPU, which the benchmark uses as the roofline denominator.  Each CTA
// writes the SM clock cycles its MMAs took.
__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, unsigned long long* cycles) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const int tid = threadIdx.x, warp = tid >> 5;
  constexpr uint32_t OFF_B = 16384, OFF_SF = OFF_B + 32768, OFF_BAR = OFF_SF + 1536;
  uint32_t* holder = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 16);
  for (uint32_t i = tid; i < OFF_SF / 4; i += 128)
    reinterpret_cast<uint32_t*>(smem)[i] = 0x30303030u | ((i * 2654435761u) & 0x07070707u);
  for (uint32_t i = tid; i < 1536 / 4; i += 128) reinterpret_cast<uint32_t*>(smem + OFF_SF)[i] = 0x7F7F7F7Fu;
  if (tid == 0) {
    mbar_init(base + OFF_BAR, 1);
    fence_mbar_init();
  }
  fence_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *holder;
  if (warp == 0) {
    const uint32_t sfa = 256 + 16, sfb = 256 + 24;
    tc_cp_sf_w(tm + sfa, smem_desc(base + OFF_SF, 128, 128, 0));
    tc_cp_sf_w(tm + sfb, smem_desc(base + OFF_SF + 512, 128, 128, 0));
    tc_cp_sf_w(tm + sfb + 4, smem_desc(base + OFF_SF + 1024, 128, 128, 0));
    const uint64_t dA = smem_desc(base, 16, 1024, 2), dB = smem_desc(base + OFF_B, 16, 1024, 2);
    tc_commit_w(base + OFF_BAR);
    bool ok = gemm_wait_raw(base + OFF_BAR, 0);
    __syncwarp();
    const unsigned long long t0 = clock64();
    for (int i = 0; ok && i < iters; i++) {
#pragma unroll
      for (int k = 0; k < 4; k++)
        mma_mxf8_ss_w(tm, dA + uint64_t(2 * k), dB + uint64_t(2 * k), idesc_mxf8(128, 256, 0, 0, k, k), tm + sfa,
                      tm + sfb, (i | k) ? 1u : 0u);
    }
    tc_commit_w(base + OFF_BAR);
    ok = gemm_wait_raw(base + OFF_BAR, 1) && ok;
    const unsigned long long t1 = clock64();
    if (!ok) atomicOr(&g_status_gemm, DEV_TIMEOUT);
    if (tid == 0) cycles[blockIdx.x] = ok ? t1 - t0 : 0ull;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

cudaError_t launch_mma_peak(int iters, int ctas, unsigned long long* cycles, cudaStream_t st) {
  constexpr int smem = 16384 + 32768 + 1536 + 64 + 1024;
  static std::atomic<unsigned long long> attr{0};
  clear_stale_error();
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (e != cudaSuccess) return e;
  mma_peak_kernel<<<unsigned(ctas), 128, smem, st>>>(iters, cycles);
  return cudaGetLastError();
}

unsigned read_status_gemm(cudaStream_t st) {
  unsigned v = 0, z = 0;
  cudaMemcpyFromSymbolAsync(&v, g_status_gemm, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
  cudaMemcpyToSymbolAsync(g_status_gemm, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
  cudaStreamSynchronize(st);
  return v;
}

}  // namespace mxfa
