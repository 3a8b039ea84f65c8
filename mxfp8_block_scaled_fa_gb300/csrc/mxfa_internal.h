// mxfa_internal.h -- host-side declarations shared by the C-ABI layer and the
// kernel translation units.  Not part of the public interface.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace mxfa {

// ---------------------------------------------------------- per-device state
// Launch attributes (the opt-in to large dynamic shared memory) and device
// properties belong to one device's context, so they are set and cached per
// device: bit d of `done` records that `fn` has succeeded on device d.
// Concurrent first calls may both run `fn`, which is idempotent.
constexpr int kMaxDevices = 64;
template <class F>
cudaError_t once_per_device(std::atomic<unsigned long long>& done, F&& fn) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return fn();
  const unsigned long long bit = 1ull << dev;
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = fn();
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Number of SMs of the current device (0 on error), cached per device.
int sm_count_current_device();

// Clears an error left by earlier runtime calls of this thread, so that the
// check after this call's launches reports only this call's own failures.
inline void clear_stale_error() { (void)cudaGetLastError(); }

// Sequence geometry.  When cu == nullptr every sequence has length `seqlen`
// and sequence g starts at token g * seqlen.
struct Seqs {
  const int32_t* cu;  // device, nseq + 1 entries (nullable)
  int nseq;
  int seqlen;   // uniform length (cu == nullptr) or maximum length
};

struct QuantArgs {
  const uint16_t* x;  // bf16 [tokens][H*D]
  int64_t tokens;
  int H, D;
  int mode;  // 0 ROW, 1 COL, 2 SQ
  Seqs seq;
  int64_t packed_tiles;
  uint8_t* data;
  uint8_t* sf_compact;  // nullable
  uint8_t* sf_packed;   // nullable
  // modes 1 and 2 only, nullable: the same input also quantized ROW (1x32
  // along D) from the same read -- payload, compact and packed scales
  uint8_t* row_data;
  uint8_t* row_sfc;
  uint8_t* row_sfp;
  // dense batches (seq.cu == nullptr) with two outputs: x as bf16
  // [tokens][H][128], box 128 x kQuantHeadsPerUnit x 32, no swizzle, for the
  // streaming kernel; has_map = 0 selects the register-staged kernels
  CUtensorMap tm_x;
  int has_map;
};
constexpr int kQuantHeadsPerUnit = 2;
cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t s);

// Lower-precision quantization (MXFP4, MXFP6, NVFP4) of bf16 x[rows][cols]
// in 1x32 (MX) or 1x16 (NVFP4) blocks along the columns; codes one per byte, or
// (MX formats) in the MMA operand form.
struct LowpArgs {
  const uint16_t* x;
  int64_t rows;
  int cols;
  int fmt;              // 0 E2M1 (MXFP4), 1 E2M3, 2 E3M2 (MXFP6), 3 NVFP4
  uint8_t* q;           // codes [rows][cols]
  int q_mma;            // MX only: q in the MMA form (16 codes packed, padded to 16 bytes)
  uint8_t* sf;          // scales [rows][cols / 32] (E8M0) or [rows][cols / 16] (E4M3)
  uint8_t* sf_packed;   // nullable, MX only: packed atoms per (128-row tile, 128-column group)
  float* tensor_scale;  // NVFP4: device fp32, receives the tensor scale
};
cudaError_t launch_lowp_quantize(const LowpArgs& a, cudaStream_t s);

struct PackArgs {
  const uint8_t* sf_compact;
  int64_t tokens;
  int H, D;
  int mode;
  Seqs seq;
  int64_t packed_tiles;
  uint8_t* sf_packed;
};
cudaError_t launch_sf_pack(const PackArgs& a, cudaStream_t s);
// Inverse of launch_sf_pack: reads a.sf_packed, writes the compact scales.
cudaError_t launch_sf_unpack(const PackArgs& a, uint8_t* sf_compact, cudaStream_t s);

struct RmsArgs {
  const uint16_t* x;
  const float* gamma;
  int64_t T;
  int C;
  float eps;
  int seg_len;
  int H, D;  // head split of C used by the packed layouts (C = H * D)
  uint8_t *row_data, *row_sfc, *row_sfp;
  uint8_t *col_data, *col_sfc, *col_sfp;
  uint8_t *sq_data, *sq_sfc, *sq_sfp;
};
cudaError_t launch_rmsnorm_quant(const RmsArgs& a, cudaStream_t s);

struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // u8 [tokens][H][128], box 128 x 1 x 128, 128B swizzle
  CUtensorMap tm_o;              // bf16 O [tokens][H][128], box 64 x 1 x 32, 128B swizzle (stores)
  const uint8_t* sfq;  // packed ROW atoms
  const uint8_t* sfk;  // packed ROW atoms
  const uint8_t* sfv;  // packed COL atoms
  Seqs sq, sk;
  int64_t total_q;
  int64_t ptiles_q, ptiles_k;  // packed tile counts (bounds of sfq / sfk, sfv)
  int H;
  float scale_log2;  // softmax scale * log2(e)
  float rescale_thr; // running max moves when it grows by more than this (log2 units)
  uint32_t p_sc_const;  // 0: P block scales from the block maxima; else this E8M0 byte for every block
  int causal;
  uint16_t* o;       // bf16 [tokens][H][128]
  uint8_t* omx;      // nullable: O quantized (ROW, 1x32 along D) E4M3 [tokens][H][128]
  uint8_t* omx_sfc;  // nullable: its compact scales [tokens][H * 4]
  uint8_t* omx_sfp;  // nullable: its packed ROW atoms (ptiles_q * H * 512 bytes)
  float* lse;
  int64_t lse_hstride;  // dense: S, varlen: total_q
  int dense_lse;        // 1: lse[(b*H + h) * S + s]; 0: lse[h * total_q + token]
  int sched_slot;       // work-counter slot of this launch (set by launch_fwd)
  int stage_o;          // 1: O leaves through TMA stores staged in the item's Q tiles (short items)
};
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t s);

struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // u8 payloads; q/do boxes 128 x 1 x 64
  CUtensorMap tm_dqacc;                 // dQ accumulator (fp32 / fp16), box 128 x 1 x 64
  CUtensorMap tm_dk, tm_dv;             // bf16 dK, dV [tokens][H][128], box 64 x 1 x 32, 128B swizzle (stores)
  const uint8_t* sfq;   // packed SQ (16 B per tile and head)
  const uint8_t* sfk;   // packed SQ
  const uint8_t* sfv;   // packed ROW atoms
  const uint8_t* sfdo;  // packed SQ
  const uint16_t* o;    // bf16
  const uint16_t* dout; // bf16
  const uint8_t* do_q;  // dO's E4M3 payload (32x32 blocks; scales sfdo)
  const float* lse;
  Seqs sq, sk;
  int64_t total_q, total_k;
  int64_t ptiles_q, ptiles_k;
  int H;
  float scale;        // softmax scale
  uint32_t p_sc_const; // 0: P^T block scales from the block maxima; else this E8M0 byte for every block
  int causal;
  int dq_mode;        // 0 fp32 accumulation, 1 fp16 with static scale
  float dq_static_scale;
  uint16_t *dq, *dk, *dv;  // bf16 outputs
  // nullable MXFP8 copies of the gradients (ROW, 1x32 along D): payload,
  // compact scales [tokens][H * 4], packed ROW atoms (dK, dV only; dQ's are
  // packed from its compact scales after the post pass)
  uint8_t *dqmx, *dqmx_sfc, *dqmx_sfp;
  uint8_t *dkmx, *dkmx_sfc, *dkmx_sfp;
  uint8_t *dvmx, *dvmx_sfc, *dvmx_sfp;
  uint8_t* rec;            // workspace: one record per (64-query tile, head)
  void* dq_acc;            // workspace [total_q][H][128] fp32 or fp16
  int64_t lse_hstride;
  int dense_lse;
  int head_group;  // dense: heads whose key tiles are scheduled together (set by launch_bwd)
};
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t s);

struct GemmArgs {
  CUtensorMap tm_a, tm_b;  // u8 [M][K/128][128] and [N][K/128][128], box 128 x 1 x 128, 128B swizzle
  const uint8_t* sfa;      // packed ROW atoms of A: entry (m / 128) * (K / 128) + k / 128
  const uint8_t* sfb;      // packed ROW atoms of B: entry (n / 128) * (K / 128) + k / 128
  int64_t M, N, K;         // multiples of 128
  int a_fmt, b_fmt;        // element format codes of the MMA kind (0 E4M3, 3 E2M3, 4 E3M2, 5 E2M1)
  uint16_t* y_bf16;        // nullable: Y bf16 [M][N]
  uint8_t *row_data, *row_sfc, *row_sfp;  // nullable: Y MXFP8, 1x32 along N
  uint8_t *col_data, *col_sfc, *col_sfp;  // nullable: Y MXFP8, 32x1 along M
};
cudaError_t launch_gemm_quant(const GemmArgs& a, cudaStream_t s);
// Tensor-pipe peak probe: `ctas` CTAs of back-to-back MMAs, cycles per CTA.
cudaError_t launch_mma_peak(int iters, int ctas, unsigned long long* cycles, cudaStream_t s);

// Read (and clear) the device status words of every kernel module.
unsigned read_status_quant(cudaStream_t s);
unsigned read_status_gemm(cudaStream_t s);
unsigned read_status_fwd(cudaStream_t s);
unsigned read_status_bwd(cudaStream_t s);

}  // namespace mxfa
