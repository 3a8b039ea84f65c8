// attn_bwd.cu -- MXFP8 block-scaled FlashAttention backward for sm_103a.
//
// What it computes ("MXFP8 FlashAttention-4 Hits 2.85 Petaflops in Meta's
// Production Training", section "Inside the TMEM Bargain and Zero-Gather
// Jagged Pipeline"; "Meta's FlashAttention-4 Achieves 2.85 PF/s with MXFP8 on
// Blackwell GPUs", item 6; "Low-Precision FlashAttention-4 ...", section
// "Hardware Adaptation for Blackwell" for the recompute):
//   five GEMMs with recompute -- S^T = K Q^T, dP^T = V dO^T, dV += P^T dO,
//   dK += dS^T Q, dQ^T = K^T dS^T -- on MXFP8 operands.  Q, K and dO carry
//   32x32 square scales, so one E4M3 payload serves both GEMM orientations;
//   V carries 1x32 scales along D.  P = exp(min(S tau - lse, 0)) is quantized
//   in 1x32 blocks along queries (the dV contraction); the min keeps P <= 1
//   when the square-block scores exceed the forward's lse.  dS = P (dP - Delta)
//   is quantized once per 32x32 block with a warp-wide absolute-maximum
//   reduction.  dQ partials are reduced into a global accumulator in FP32, or
//   in FP16 after multiplying by a static power-of-two scale.  dQ, dK, dV are
//   written as bf16 and, on request, also as MXFP8 (1x32 along D).
//
// Structure: one CTA = one 128-key tile of one head, looping over 64-query
// tiles (16 warps, 1 CTA per SM; dense non-causal grids run heads in groups
// so that their fp32 dQ rows stay in L2):
//   warp 0       TMA producer: K, V (+ V scale atom) once; ring of Q_i, dO_i
//                and the tile records made by the preparation kernel
//   warp 1       TMEM owner + MMA issuer for S^T and dP^T
//   warps 2-3    key-tile scale atoms (K, rows = keys and rows = d); warp 2
//                then issues the gradient GEMMs (dV, dK, dQ^T)
//   warps 4-11   P / dS: thread = key row, warpgroup 0 queries 0-31,
//                warpgroup 1 queries 32-63 of the tile
//   warps 12-15  dQ drain: TMEM dQ^T -> shared -> one tiled TMA reduce-add
// Scale atoms enter TMEM by tcgen05.cp, issued by the MMA issuer that reads them.
// TMEM columns: dV [0,128) dK [128,256) S^T [256,320) dP^T [320,384)
//               dQ^T [384,448) scale slots [448,512).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "mx_ptx.cuh"
#include "mx_seq.cuh"
#include "mxfa_internal.h"

namespace mxfa {

static __device__ unsigned g_status_bwd;

namespace bwd {
constexpr int KT = 128;                 // keys per CTA
constexpr int QT = 64;                  // queries per inner tile
constexpr int NSQ = 4;                  // Q / dO / tile-record ring stages
// Per (64-query tile, head) record written by the preparation kernel:
// four scale atoms (Q and dO, rows = queries; dO and Q, rows = d) and the
// tile's -lse * log2(e) and -Delta (negated so that each enters one FMA / add).
constexpr int REC_SFQ = 0, REC_SFDO = 512, REC_SFDOT = 1024, REC_SFQT = 1536, REC_NL2 = 2048,
              REC_NDELTA = 2304, REC_BYTES = 2560;
constexpr int KV_BYTES = KT * 128;      // 16 KB
constexpr int QD_BYTES = QT * 128;      // 8 KB
constexpr int PS_BYTES = KT * QT;       // 8 KB (128 rows x 64 B)

constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + KV_BYTES;
constexpr int OFF_Q = OFF_V + KV_BYTES;                 // NSQ stages
constexpr int OFF_DO = OFF_Q + NSQ * QD_BYTES;          // NSQ stages
constexpr int OFF_PT = OFF_DO + NSQ * QD_BYTES;         // 2 buffers, SW64
constexpr int OFF_DST = OFF_PT + 2 * PS_BYTES;          // 2 buffers, SW64
constexpr int DQS_BYTES = QT * 512;                    // one dQ staging tile (fp32)
constexpr int OFF_DQS = OFF_DST + 2 * PS_BYTES;         // dQ staging, 2 tiles
constexpr int OFF_REC = OFF_DQS + 2 * DQS_BYTES;       // NSQ tile records
constexpr int OFF_ATOM = OFF_REC + NSQ * REC_BYTES;
// scale atoms (512 B each)
constexpr int A_SFK = 0, A_SFV = 1, A_SFKT = 2;
constexpr int A_SFPT = 3, A_SFDST = A_SFPT + 2, A_SFDS = A_SFDST + 2;  // x2
constexpr int NATOM = A_SFDS + 2;
constexpr int OFF_BAR = OFF_ATOM + NATOM * 512;
enum {
  B_KVFULL = 0, B_KCONST, B_QDOFULL, B_QDOEMPTY = B_QDOFULL + NSQ,
  B_SDPFULL = B_QDOEMPTY + NSQ, B_SDPFREE, B_PATOM, B_PDSEMPTY = B_PATOM + 2,
  B_DQFULL = B_PDSEMPTY + 2, B_DQEMPTY, B_KVDONE, B_TEAR, B_TEAR2, NBAR
};
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "backward tile exceeds the shared memory of one CTA");
// the dK / dV epilogue stages 8 x 4 KB of 128B-swizzled rows in the Q ring
static_assert(OFF_Q % 1024 == 0 && OFF_DO == OFF_Q + NSQ * QD_BYTES && 2 * NSQ * QD_BYTES >= 8 * 8192,
              "dK / dV staging does not fit the Q and dO rings");

constexpr uint32_t COL_DV = 0, COL_DK = 128, COL_S = 256, COL_DP = 320, COL_DQ = 384;
constexpr uint32_t COL_SFK = 448, COL_SFV = 452, COL_SFKT = 456, COL_SFQ = 460, COL_SFDO = 464,
                   COL_SFPT = 468, COL_SFDOT = 476, COL_SFDST = 484, COL_SFQT = 492,
                   COL_SFDS = 500;  // the last five are x2 (tile parity), 4 columns each
constexpr int NTHREADS = 512;
}  // namespace bwd

// ------------------------------------------------------------ pre / post
// Tile records.  One CTA (256 threads) per (64-query tile of a sequence, head):
//   -Delta[r] with Delta[r] = sum_d dO^[r,d] * O[r,d] (fp32, warp per row), dO^
//   the dequantized 32x32-block dO that also enters dP = dO^ V^, so that
//   dS = P (dP - Delta) cancels consistently on peaked softmax rows,
//   -lse[r] * log2(e)  (-inf past the sequence end: P = 2^-inf = 0),
//   the four scale atoms of the tile built from the packed square scales of
//   Q and dO: rows = queries (for S^T and dP^T) and rows = d (for dK and dV).
// Atom word w (bytes 4w..4w+3) holds row (w & 3) * 32 + (w >> 2), k-blocks
// 0..3 in its bytes; a square-scale entry holds byte 4 * tb + db.
__global__ void __launch_bounds__(256) bwd_prep_kernel(BwdArgs a) {
  using namespace bwd;
  const int t = blockIdx.x, h = blockIdx.y, g = blockIdx.z;
  int64_t s0;
  int L;
  seq_info(a.sq, g, s0, L);
  const int esz = a.dq_mode == 1 ? 2 : 4;
  // zero dQ accumulator rows [r0, r1) of head h (16-byte chunks)
  auto zero_rows = [&](int64_t r0, int64_t r1) {
    const int chunks = 128 * esz / 16;
    for (int64_t i = threadIdx.x; i < (r1 - r0) * chunks; i += 256) {
      uint8_t* row = reinterpret_cast<uint8_t*>(a.dq_acc) + ((r0 + i / chunks) * a.H + h) * 128 * esz;
      *reinterpret_cast<uint4*>(row + 16 * (i % chunks)) = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  // tokens outside every sequence (before the first, after the last) get dQ = 0
  if (a.sq.cu != nullptr && t == 0) {
    if (g == 0) zero_rows(0, __ldg(a.sq.cu));
    if (g == a.sq.nseq - 1) zero_rows(__ldg(a.sq.cu + a.sq.nseq), a.total_q);
  }
  if (t * QT >= L) return;
  const int64_t t128 = seq_units_before_warp(a.sq, g, 128, threadIdx.x & 31) + t / 2;
  if (t128 >= a.ptiles_q) {
    atomicOr(&g_status_bwd, DEV_BAD_INDEX);
    return;
  }
  uint8_t* rec = a.rec + ((seq_units_before_warp(a.sq, g, QT, threadIdx.x & 31) + t) * a.H + h) * REC_BYTES;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint4 q4 = __ldg(reinterpret_cast<const uint4*>(a.sfq + (t128 * a.H + h) * 16));
  const uint4 d4 = __ldg(reinterpret_cast<const uint4*>(a.sfdo + (t128 * a.H + h) * 16));
  auto pick = [](uint4 e, int tb) { return tb == 0 ? e.x : tb == 1 ? e.y : tb == 2 ? e.z : e.w; };
  const int tb0 = (t & 1) * 2;
  float* ndelta = reinterpret_cast<float*>(rec + REC_NDELTA);
  // the warp's eight rows: every load in flight first, then the dot products
  uint2 ov[8];
  uint32_t dq4[8];
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const int q = t * QT + warp * 8 + i;
    ov[i] = make_uint2(0u, 0u);
    dq4[i] = 0u;
    if (q < L) {
      const int64_t off = ((s0 + q) * a.H + h) * 128 + lane * 4;
      ov[i] = *reinterpret_cast<const uint2*>(a.o + off);
      dq4[i] = *reinterpret_cast<const uint32_t*>(a.do_q + off);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const int r = warp * 8 + i;
    // dO^ of these four columns: E4M3 codes times the 32x32 block scale of
    // (query block tb0 + r / 32, d block lane / 8); rows past the sequence
    // hold zeros
    const uint32_t sb = (pick(d4, tb0 + (r >> 5)) >> (8 * (lane >> 3))) & 0xFFu;
    const float f = e8m0_value(sb);
    const float2 d01 = e4m3x2_to_float2(dq4[i] & 0xFFFFu), d23 = e4m3x2_to_float2(dq4[i] >> 16);
    auto lo = [](uint32_t w) { return __uint_as_float(w << 16); };
    auto hi = [](uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); };
    float d = lo(ov[i].x) * (d01.x * f) + hi(ov[i].x) * (d01.y * f) + lo(ov[i].y) * (d23.x * f) +
              hi(ov[i].y) * (d23.y * f);
#pragma unroll
    for (int off2 = 16; off2 >= 1; off2 >>= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, off2);
    if (lane == 0) ndelta[r] = -d;
  }
  // the dQ accumulator rows of this tile start at zero (each token row of a
  // sequence belongs to exactly one (64-query tile, head))
  zero_rows(s0 + t * QT, s0 + t * QT + min(QT, L - t * QT));
  if (tid < QT) {
    const int q = t * QT + tid;
    float nl2 = -INFINITY;  // rows past the sequence: P = 2^-inf = 0
    if (q < L) {
      const float lse = a.dense_lse ? a.lse[(int64_t(g) * a.H + h) * a.lse_hstride + q]
                                    : a.lse[int64_t(h) * a.lse_hstride + s0 + q];
      nl2 = -(lse * 1.4426950408889634f);
    }
    reinterpret_cast<float*>(rec + REC_NL2)[tid] = nl2;
  }
  if (tid < 128) {
    const int w = tid, rg = w & 3;
    uint32_t* aq = reinterpret_cast<uint32_t*>(rec + REC_SFQ);
    uint32_t* ad = reinterpret_cast<uint32_t*>(rec + REC_SFDO);
    aq[w] = rg < 2 ? pick(q4, tb0 + rg) : 0x7F7F7F7Fu;   // rows = queries, k = d-blocks
    ad[w] = rg < 2 ? pick(d4, tb0 + rg) : 0x7F7F7F7Fu;
  } else {
    const int w = tid - 128, rg = w & 3;               // rows = d (block rg), k = query blocks
    const uint32_t sh = 8u * uint32_t(rg);
    uint32_t* aqt = reinterpret_cast<uint32_t*>(rec + REC_SFQT);
    uint32_t* adt = reinterpret_cast<uint32_t*>(rec + REC_SFDOT);
    aqt[w] = ((pick(q4, tb0) >> sh) & 0xFFu) | (((pick(q4, tb0 + 1) >> sh) & 0xFFu) << 8) | 0x7F7F0000u;
    adt[w] = ((pick(d4, tb0) >> sh) & 0xFFu) | (((pick(d4, tb0 + 1) >> sh) & 0xFFu) << 8) | 0x7F7F0000u;
  }
}

// dQ = bf16(acc * mult) as below, and the same bf16 dQ as MXFP8: one thread
// per 1x32 block along D (the flat element index / 32 is the block's index
// in the compact [tokens][H * 4] scale layout).
__global__ void __launch_bounds__(256) bwd_post_mx_kernel(const void* __restrict__ acc,
                                                          uint16_t* __restrict__ dq, int64_t n, int mode,
                                                          float mult, uint8_t* __restrict__ dqmx,
                                                          uint8_t* __restrict__ dqmx_sfc) {
  const int64_t blk = int64_t(blockIdx.x) * 256 + threadIdx.x;
  const int64_t i = blk * 32;
  if (i >= n) return;
  uint32_t w[16];
#pragma unroll
  for (int q8 = 0; q8 < 4; q8++) {
    float v[8];
    if (mode == 0) {
      const float4 x = *reinterpret_cast<const float4*>(static_cast<const float*>(acc) + i + 8 * q8);
      const float4 y = *reinterpret_cast<const float4*>(static_cast<const float*>(acc) + i + 8 * q8 + 4);
      v[0] = x.x * mult; v[1] = x.y * mult; v[2] = x.z * mult; v[3] = x.w * mult;
      v[4] = y.x * mult; v[5] = y.y * mult; v[6] = y.z * mult; v[7] = y.w * mult;
    } else {
      const uint4 x = *reinterpret_cast<const uint4*>(static_cast<const __half*>(acc) + i + 8 * q8);
      const uint32_t hw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw[j]));
        v[2 * j] = f.x * mult;
        v[2 * j + 1] = f.y * mult;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; j++) {
      __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
      w[4 * q8 + j] = *reinterpret_cast<uint32_t*>(&p);
    }
    *reinterpret_cast<uint4*>(dq + i + 8 * q8) = make_uint4(w[4 * q8], w[4 * q8 + 1], w[4 * q8 + 2], w[4 * q8 + 3]);
  }
  const uint32_t sc = mx_block_e8m0(w);
  mx_block_store(dqmx + i, w, sc);
  if (dqmx_sfc != nullptr) dqmx_sfc[blk] = uint8_t(sc);
}

// dQ = bf16(acc * mult): acc is fp32 holding unscaled sums (mode 0, mult =
// softmax scale) or fp16 holding scale * static_scale times them (mode 1,
// mult = 1 / static_scale).
__global__ void __launch_bounds__(256) bwd_post_kernel(const void* __restrict__ acc,
                                                       uint16_t* __restrict__ dq, int64_t n,
                                                       int mode, float mult) {
  const int64_t i = (int64_t(blockIdx.x) * 256 + threadIdx.x) * 8;
  if (i >= n) return;
  float v[8];
  if (mode == 0) {
    const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(acc) + i);
    const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(acc) + i + 4);
    v[0] = a.x * mult; v[1] = a.y * mult; v[2] = a.z * mult; v[3] = a.w * mult;
    v[4] = b.x * mult; v[5] = b.y * mult; v[6] = b.z * mult; v[7] = b.w * mult;
  } else {
    const uint4 a = *reinterpret_cast<const uint4*>(static_cast<const __half*>(acc) + i);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
      v[2 * j] = f.x * mult;
      v[2 * j + 1] = f.y * mult;
    }
  }
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; j++) {
    __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
    w[j] = *reinterpret_cast<uint32_t*>(&p);
  }
  *reinterpret_cast<uint4*>(dq + i) = make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float bex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ bool bwait_raw(uint32_t bar, uint32_t parity) {
  unsigned long long t0 = global_ns();
  while (!mbar_try_wait_sleep(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}
// One arrival for the whole warp, after every lane's prior work (each lane
// fences its own tcgen05 / shared-memory writes before calling this).
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}
// Warp-uniform bounded wait (all lanes agree on the outcome).
__device__ __forceinline__ bool wwait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag, &g_status_bwd));
}
// Byte offset of 16-byte chunk c of row r in a 64-byte-row, 64B-swizzled tile.
__device__ __forceinline__ uint32_t sw64(int r, int c) {
  return uint32_t(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

// ------------------------------------------------------------------ main
__global__ void __launch_bounds__(bwd::NTHREADS, 1) attn_bwd_kernel(const __grid_constant__ BwdArgs a) {
  using namespace bwd;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- work item: (sequence g, head h, key tile kt)
  int g, h, kt;
  if (a.sk.cu == nullptr) {
    // dense: heads in groups of head_group, whose key tiles run together so
    // that the dQ accumulator rows they reduce into stay in L2; inside a
    // group, heavy (early, causal) key tiles first (causal runs use a single
    // group: key tile major over all heads)
    const int per = a.H * a.sk.nseq;
    const int nkt = (a.sk.seqlen + KT - 1) / KT;
    const int G = a.head_group;
    const int gi = int(blockIdx.x) / (G * nkt), i = int(blockIdx.x) % (G * nkt);
    const int gc = min(G, per - gi * G);
    kt = i / gc;
    const int bh = gi * G + i % gc;
    g = bh / a.H;
    h = bh % a.H;
  } else {
    kt = blockIdx.x;
    h = blockIdx.y;
    g = blockIdx.z;
  }
  int64_t sq0, sk0;
  int lq, lk;
  seq_info(a.sq, g, sq0, lq);
  seq_info(a.sk, g, sk0, lk);
  if (kt * KT >= lk) return;
  const int nq = (lq + QT - 1) / QT;
  const int first = a.causal ? min(nq, (kt * KT) / QT) : 0;
  const int ntile = nq - first;
  const int64_t tq_base = seq_units_before_warp(a.sq, g, 128, lane);
  const int64_t tq64 = seq_units_before_warp(a.sq, g, QT, lane);  // first tile record of this sequence
  const int64_t tk = seq_units_before_warp(a.sk, g, 128, lane) + kt;

  const uint32_t bar0 = base + OFF_BAR;
  auto BAR = [&](int i) { return bar0 + 8u * uint32_t(i); };
  auto ATOM = [&](int i) { return smem + OFF_ATOM + 512 * i; };
  auto ATOMA = [&](int i) { return base + OFF_ATOM + 512u * uint32_t(i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 8);

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(BAR(B_KVFULL), 1);
    mbar_init(BAR(B_KCONST), 2);  // arrivals are one per warp
    for (int s = 0; s < NSQ; s++) {
      mbar_init(BAR(B_QDOFULL + s), 1);
      mbar_init(BAR(B_QDOEMPTY + s), 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(BAR(B_PATOM + b), 8);   // P / dS warps
      mbar_init(BAR(B_PDSEMPTY + b), 1);
    }
    mbar_init(BAR(B_SDPFULL), 1);
    mbar_init(BAR(B_SDPFREE), 8);
    mbar_init(BAR(B_DQFULL), 1);
    mbar_init(BAR(B_DQEMPTY), 4);
    mbar_init(BAR(B_KVDONE), 1);
    mbar_init(BAR(B_TEAR), 1);
    mbar_init(BAR(B_TEAR2), 1);
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
  const bool bad = tk >= a.ptiles_k || tq_base + (lq + 127) / 128 > a.ptiles_q;
  if (bad && tid == 0) {
    atomicOr(&g_status_bwd, DEV_BAD_INDEX);
    *abort_flag = 1;
  }
  __syncthreads();

  if (bad) {
    // nothing issued; fall through to teardown
  } else if (warp == 0) {
    warp_converged();
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&a.tm_q);
      tma_prefetch_desc(&a.tm_k);
      tma_prefetch_desc(&a.tm_v);
      tma_prefetch_desc(&a.tm_do);
      mbar_arrive_expect_tx(BAR(B_KVFULL), 2 * KV_BYTES + 512);
      const int krow = int(sk0 + int64_t(kt) * KT);
      tma_load_3d(base + OFF_K, &a.tm_k, BAR(B_KVFULL), 0, h, krow);
      tma_load_3d(base + OFF_V, &a.tm_v, BAR(B_KVFULL), 0, h, krow);
      bulk_load(ATOMA(A_SFV), a.sfv + (tk * a.H + h) * 512, 512, BAR(B_KVFULL));
      int issued = 0;
      for (int ii = 0; ii < ntile; ii++) {
        const int s = ii % NSQ, i = first + ii;
        if (ii >= NSQ && !mbar_wait(BAR(B_QDOEMPTY + s), ((ii / NSQ) - 1) & 1, abort_flag, &g_status_bwd))
          break;
        issued = ii + 1;
        const uint32_t fb = BAR(B_QDOFULL + s);
        mbar_arrive_expect_tx(fb, 2 * QD_BYTES + REC_BYTES);
        const int qrow = int(sq0 + int64_t(i) * QT);
        tma_load_3d(base + OFF_Q + s * QD_BYTES, &a.tm_q, fb, 0, h, qrow);
        tma_load_3d(base + OFF_DO + s * QD_BYTES, &a.tm_do, fb, 0, h, qrow);
        bulk_load(base + OFF_REC + s * REC_BYTES, a.rec + ((tq64 + i) * a.H + h) * REC_BYTES,
                  REC_BYTES, fb);
      }
      for (int ii = max(0, issued - NSQ); ii < issued; ii++)
        bwait_raw(BAR(B_QDOFULL + ii % NSQ), (ii / NSQ) & 1);
      bwait_raw(BAR(B_KVFULL), 0);
    }
  } else if (warp == 2 || warp == 3) {
    warp_converged();
    // ------------------------------------------------ key-tile scale atoms
    // Atom word w (bytes 4w..4w+3) holds row r = (w & 3) * 32 + (w >> 2),
    // k-blocks 0..3 in its bytes.  Square scale entry: byte 4 * tb + db.
    const int t = tid - 64;
    const uint4 k4 = __ldg(reinterpret_cast<const uint4*>(a.sfk + (tk * a.H + h) * 16));
    // word tb of an entry holds the bytes of token block tb for d-blocks 0..3
    auto pick = [](uint4 e, int tb) {
      return tb == 0 ? e.x : tb == 1 ? e.y : tb == 2 ? e.z : e.w;
    };
    // byte db of token blocks tb0, tb0+1 (and tb0+2, tb0+3 when all4), padding 0x7F
    auto col_bytes = [&](uint4 e, int db, int tb0, bool all4) {
      const uint32_t sh = 8u * uint32_t(db);
      const uint32_t b0 = (pick(e, tb0) >> sh) & 0xFFu, b1 = (pick(e, tb0 + 1) >> sh) & 0xFFu;
      const uint32_t b2 = all4 ? (e.z >> sh) & 0xFFu : 0x7Fu, b3 = all4 ? (e.w >> sh) & 0xFFu : 0x7Fu;
      return b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
    };
    for (int w = t; w < 128; w += 64) {
      reinterpret_cast<uint32_t*>(ATOM(A_SFK))[w] = pick(k4, w & 3);                 // rows = keys
      reinterpret_cast<uint32_t*>(ATOM(A_SFKT))[w] = col_bytes(k4, w & 3, 0, true);  // rows = d
    }
    warp_arrive(BAR(B_KCONST), lane);
    if (warp == 2) {
      warp_converged();
      // -------------------------------------- MMA issuer: dV, dK, dQ^T
      // The whole warp walks the schedule; every tcgen05 operation is issued
      // through a lane elected inside the instruction.
      const uint32_t tm = __shfl_sync(0xFFFFFFFFu, tmem, 0);
      auto wait_all = [&](uint32_t bar, uint32_t par) {
        return __all_sync(0xFFFFFFFFu, mbar_wait(bar, par, abort_flag, &g_status_bwd));
      };
      // scale atom (512 bytes in shared memory) -> TMEM slot, replicated to the
      // four lane quadrants; ordered before this thread's later MMAs
      auto cp_sf = [&](uint32_t col, uint32_t saddr) {
        tc_cp_sf_w(tm + col, smem_desc(saddr, 128, 128, 0));
      };
      const uint64_t dK_mn = smem_desc(base + OFF_K, 8192, 1024, 2);    // K^T, MN-major (dQ^T A)
      // K (shared memory) and the K^T scale atom
      bool ok = wait_all(BAR(B_KVFULL), 0) && wait_all(BAR(B_KCONST), 0);
      tc_fence_after();
      cp_sf(COL_SFKT, ATOMA(A_SFKT));
      // dV += P^T dO, dK += dS^T Q, dQ^T = K^T dS^T for local tile jj
      auto grads = [&](int jj) -> bool {
        const int s = jj % NSQ, b = jj & 1;
        // P^T, dS^T and their scale atoms written; the tile record in place;
        // the dQ^T accumulator drained
        if (!wait_all(BAR(B_QDOFULL + s), (jj / NSQ) & 1) || !wait_all(BAR(B_PATOM + b), (jj >> 1) & 1))
          return false;
        tc_fence_after();
        // slot b was last read by tile jj - 2's MMAs, earlier in this stream
        const uint32_t rec = base + OFF_REC + s * REC_BYTES;
        cp_sf(COL_SFPT + 4 * b, ATOMA(A_SFPT + b));
        cp_sf(COL_SFDOT + 4 * b, rec + REC_SFDOT);
        cp_sf(COL_SFDST + 4 * b, ATOMA(A_SFDST + b));
        cp_sf(COL_SFQT + 4 * b, rec + REC_SFQT);
        cp_sf(COL_SFDS + 4 * b, ATOMA(A_SFDS + b));
        const uint64_t dPt = smem_desc(base + OFF_PT + b * PS_BYTES, 16, 512, 4);
        const uint64_t dSt_k = smem_desc(base + OFF_DST + b * PS_BYTES, 16, 512, 4);
        const uint64_t dSt_mn = smem_desc(base + OFF_DST + b * PS_BYTES, 8192, 512, 4);
        const uint64_t dQ_mn = smem_desc(base + OFF_Q + s * QD_BYTES, 8192, 1024, 2);
        const uint64_t dDO_mn = smem_desc(base + OFF_DO + s * QD_BYTES, 8192, 1024, 2);
#pragma unroll
        for (int k = 0; k < 2; k++) {
          const uint32_t acc = (jj > 0 || k > 0) ? 1u : 0u;
          mma_mxf8_ss_w(tm + COL_DV, dPt + uint64_t(2 * k), dDO_mn + uint64_t(256 * k),
                        idesc_mxf8(128, 128, 0, 1, k, k), tm + COL_SFPT + 4 * b, tm + COL_SFDOT + 4 * b,
                        acc);
          mma_mxf8_ss_w(tm + COL_DK, dSt_k + uint64_t(2 * k), dQ_mn + uint64_t(256 * k),
                        idesc_mxf8(128, 128, 0, 1, k, k), tm + COL_SFDST + 4 * b, tm + COL_SFQT + 4 * b,
                        acc);
        }
        tc_commit_w(BAR(B_QDOEMPTY + s));  // Q_j and dO_j are no longer read
        // dQ^T reuses one accumulator: the previous tile's must have been drained
        if (jj >= 1 && !wait_all(BAR(B_DQEMPTY), (jj - 1) & 1)) return false;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; k++)
          mma_mxf8_ss_w(tm + COL_DQ, dK_mn + uint64_t(256 * k), dSt_mn + uint64_t(128 * k),
                        idesc_mxf8(128, 64, 1, 1, k, k), tm + COL_SFKT, tm + COL_SFDS + 4 * b,
                        k > 0 ? 1u : 0u);
        tc_commit_w(BAR(B_PDSEMPTY + b));
        tc_commit_w(BAR(B_DQFULL));
        return true;
      };
      for (int jj = 0; ok && jj < ntile; jj++) ok = grads(jj);
      tc_commit_w(BAR(B_KVDONE));
      tc_commit_w(BAR(B_TEAR2));
      bwait_raw(BAR(B_TEAR2), 0);
      __syncwarp();
    }
  } else if (warp == 1) {
    warp_converged();
    // ------------------------------------------------ MMA issuer: S^T, dP^T
    // The whole warp walks the schedule (descriptors and TMEM addresses are
    // warp-uniform) and issues every tcgen05 operation through a lane elected
    // inside the instruction.  Scale atoms enter TMEM by tcgen05.cp in the same stream as the MMAs
    // that read them (replicated 32x128b x4 layout: lane L, column c holds
    // rows 32c + L % 32, k-blocks in its bytes).
    // The gradient GEMMs have an issuer of their own (warp 2): tcgen05.mma
    // issue stalls while the tensor pipe's queue is full, and an issuing warp
    // shares its SM sub-partition with arithmetic-heavy warps, so two
    // independent issue streams keep the pipe fed better than one.
    {
      const uint32_t tm = __shfl_sync(0xFFFFFFFFu, tmem, 0);
      auto wait_all = [&](uint32_t bar, uint32_t par) {
        return __all_sync(0xFFFFFFFFu, mbar_wait(bar, par, abort_flag, &g_status_bwd));
      };
      // descriptor bases (start-address field advanced by byte offset >> 4)
      const uint64_t dK_k = smem_desc(base + OFF_K, 16, 1024, 2);       // K, K-major (S^T A)
      const uint64_t dV_k = smem_desc(base + OFF_V, 16, 1024, 2);       // V, K-major (dP^T A)
      auto cp_sf = [&](uint32_t col, uint32_t saddr) {
        tc_cp_sf_w(tm + col, smem_desc(saddr, 128, 128, 0));
      };
      bool ok = wait_all(BAR(B_KVFULL), 0) && wait_all(BAR(B_KCONST), 0);
      tc_fence_after();
      cp_sf(COL_SFK, ATOMA(A_SFK));
      cp_sf(COL_SFV, ATOMA(A_SFV));
      for (int ii = 0; ok && ii < ntile; ii++) {
        const int s = ii % NSQ;
        // completion ii of SDPFREE: the S^T / dP^T columns are free
        if (!wait_all(BAR(B_QDOFULL + s), (ii / NSQ) & 1) || !wait_all(BAR(B_SDPFREE), ii & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // this tile's Q / dO scales; the slots were last read by the previous
        // tile's MMAs, earlier in this stream
        cp_sf(COL_SFQ, base + OFF_REC + s * REC_BYTES + REC_SFQ);
        cp_sf(COL_SFDO, base + OFF_REC + s * REC_BYTES + REC_SFDO);
        const uint64_t dQ_k = smem_desc(base + OFF_Q + s * QD_BYTES, 16, 1024, 2);
        const uint64_t dDO_k = smem_desc(base + OFF_DO + s * QD_BYTES, 16, 1024, 2);
#pragma unroll
        for (int k = 0; k < 4; k++)
          mma_mxf8_ss_w(tm + COL_S, dK_k + uint64_t(2 * k), dQ_k + uint64_t(2 * k),
                        idesc_mxf8(128, 64, 0, 0, k, k), tm + COL_SFK, tm + COL_SFQ, k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 4; k++)
          mma_mxf8_ss_w(tm + COL_DP, dV_k + uint64_t(2 * k), dDO_k + uint64_t(2 * k),
                        idesc_mxf8(128, 64, 0, 0, k, k), tm + COL_SFV, tm + COL_SFDO, k > 0 ? 1u : 0u);
        tc_commit_w(BAR(B_SDPFULL));
      }
      // every MMA of this issuer has completed before TMEM is released
      tc_commit_w(BAR(B_TEAR));
      bwait_raw(BAR(B_TEAR), 0);
      __syncwarp();
    }
  } else if (warp >= 4 && warp < 12) {
    warp_converged();
    // ------------------------------------------------------------ P / dS
    // Load S^T and dP^T of the tile from TMEM, free their columns, form and
    // quantize P and dS, store P^T / dS^T (shared memory, the gradient GEMMs'
    // A / B operands) and the scale bytes of the three computed scale atoms,
    // then signal the gradient issuer.  No barrier among these warps.
    const int hq = (warp - 4) >> 2;            // query half of the tile
    const int r = (warp & 3) * 32 + lane;      // key row = TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const int kpos = kt * KT + r;
    const bool kvalid = kpos < lk;
    const float sl2 = a.scale * 1.4426950408889634f;
    warp_arrive(BAR(B_SDPFREE), lane);  // completion 0: S^T / dP^T columns free
    bool ok = true;
    for (int ii = 0; ii < ntile; ii++) {
      const int i = first + ii, b = ii & 1, s = ii % NSQ;
      float sv[32], dp[32];
      float pmax = 0.0f;
      uint32_t pw[8], dw[8];
      uint32_t sp = 0, sd = 0;
      if (!wwait(BAR(B_SDPFULL), ii & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      tmem_ld32(tmem + lane_base + COL_S + 32 * hq, reinterpret_cast<uint32_t*>(sv));
      tmem_ld32(tmem + lane_base + COL_DP + 32 * hq, reinterpret_cast<uint32_t*>(dp));
      // the tile's record and the P^T / dS^T buffer are nearly always ready by
      // now: test both while the loads are in flight, wait only if needed
      const bool rec_ready = mbar_test(BAR(B_QDOFULL + s), (ii / NSQ) & 1);
      const bool buf_ready = ii < 2 || mbar_test(BAR(B_PDSEMPTY + b), ((ii >> 1) - 1) & 1);
      tmem_wait_ld();
      reg_fence32(reinterpret_cast<uint32_t*>(sv));
      reg_fence32(reinterpret_cast<uint32_t*>(dp));
      tc_fence_before();
      warp_arrive(BAR(B_SDPFREE), lane);  // completion ii + 1
      // -lse * log2 e and -Delta of the tile, from the stage's record
      if (!__all_sync(0xFFFFFFFFu, rec_ready) && !wwait(BAR(B_QDOFULL + s), (ii / NSQ) & 1, abort_flag)) {
        ok = false;
        break;
      }
      const uint8_t* rec = smem + OFF_REC + s * REC_BYTES;
      {
        // per query of this half: -lse log2 e and -Delta, four queries per 16-byte load
        const float4* nl4 = reinterpret_cast<const float4*>(rec + REC_NL2) + 8 * hq;
        const float4* nd4 = reinterpret_cast<const float4*>(rec + REC_NDELTA) + 8 * hq;
        const int q0 = i * QT + 32 * hq;
        // keys past the sequence and (causal) keys after the query: S = -inf,
        // so that P = 2^-inf = 0 and dS = 0; only tiles on the edge need it
        if (__any_sync(0xFFFFFFFFu, !kvalid || (a.causal && kpos > q0))) {
#pragma unroll
          for (int c = 0; c < 32; c++)
            if (!kvalid || (a.causal && kpos > q0 + c)) sv[c] = -INFINITY;
        }
        const float2 sl2v = make_float2(sl2, sl2);
        // exponent arguments t = fl(S * fl(scale * log2 e) - lse * log2 e)
        float tmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 n = nl4[c / 4];
          const float2 t0 = ffma2(make_float2(sv[c], sv[c + 1]), sl2v, make_float2(n.x, n.y));
          const float2 t1 = ffma2(make_float2(sv[c + 2], sv[c + 3]), sl2v, make_float2(n.z, n.w));
          sv[c] = t0.x;
          sv[c + 1] = t0.y;
          sv[c + 2] = t1.x;
          sv[c + 3] = t1.y;
          tmax = fmax3(tmax, t0.x, t0.y);
          tmax = fmax3(tmax, t1.x, t1.y);
        }
        // P <= 1: exact attention has S * scale <= lse, but S recomputed from
        // the square-block operands can exceed the forward's lse (by hundreds
        // when outliers meet coarse shared scales), so t is clamped at 0
        if (tmax > 0.0f) {
#pragma unroll
          for (int c = 0; c < 32; c++) sv[c] = fminf(sv[c], 0.0f);
          tmax = 0.0f;
        }
        float damax = 0.0f;
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          // P = 2^t, dS = P * (dP - Delta)
          const float4 nd = nd4[c / 4];
          const float2 ndc = (c & 2) ? make_float2(nd.z, nd.w) : make_float2(nd.x, nd.y);
          const float p0 = bex2(sv[c]), p1 = bex2(sv[c + 1]);
          const float2 ds = fmul2(make_float2(p0, p1), fadd2(make_float2(dp[c], dp[c + 1]), ndc));
          sv[c] = p0;
          sv[c + 1] = p1;
          dp[c] = ds.x;
          dp[c + 1] = ds.y;
          damax = fmax3(damax, fabsf(ds.x), fabsf(ds.y));
        }
        // the largest P of this thread's block (2^t is monotone in t)
        pmax = bex2(tmax);
        // P^T: one 1x32 block along queries per thread; dS: one 32x32 block
        // per warp, its maximum by a warp-wide absolute-maximum reduction
        float wmax;
        asm volatile("redux.sync.max.abs.f32 %0, %1, 0xffffffff;" : "=f"(wmax) : "f"(damax));
        sp = a.p_sc_const ? a.p_sc_const : e8m0_from_amax(pmax);
        sd = e8m0_from_amax(wmax);
        const float2 ip = make_float2(e8m0_inv_scale(sp), e8m0_inv_scale(sp));
        const float2 id = make_float2(e8m0_inv_scale(sd), e8m0_inv_scale(sd));
#pragma unroll
        for (int c = 0; c < 8; c++) {
          const float2 p01 = fmul2(make_float2(sv[4 * c], sv[4 * c + 1]), ip);
          const float2 p23 = fmul2(make_float2(sv[4 * c + 2], sv[4 * c + 3]), ip);
          const float2 d01 = fmul2(make_float2(dp[4 * c], dp[4 * c + 1]), id);
          const float2 d23 = fmul2(make_float2(dp[4 * c + 2], dp[4 * c + 3]), id);
          pw[c] = cvt_e4m3x2(p01.x, p01.y) | (cvt_e4m3x2(p23.x, p23.y) << 16);
          dw[c] = cvt_e4m3x2(d01.x, d01.y) | (cvt_e4m3x2(d23.x, d23.y) << 16);
        }
      }
      if (!__all_sync(0xFFFFFFFFu, buf_ready) && !wwait(BAR(B_PDSEMPTY + b), ((ii >> 1) - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      {
        uint8_t* pt = smem + OFF_PT + b * PS_BYTES;
        uint8_t* dst = smem + OFF_DST + b * PS_BYTES;
        *reinterpret_cast<uint4*>(pt + sw64(r, 2 * hq)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        *reinterpret_cast<uint4*>(pt + sw64(r, 2 * hq + 1)) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
        *reinterpret_cast<uint4*>(dst + sw64(r, 2 * hq)) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
        *reinterpret_cast<uint4*>(dst + sw64(r, 2 * hq + 1)) = make_uint4(dw[4], dw[5], dw[6], dw[7]);
        const int aoff = (r & 31) * 16 + (r >> 5) * 4 + hq;      // row = key, k-block = query half
        ATOM(A_SFPT + b)[aoff] = uint8_t(sp);
        ATOM(A_SFDST + b)[aoff] = uint8_t(sd);
        ATOM(A_SFDS + b)[lane * 16 + hq * 4 + (warp & 3)] = uint8_t(sd);  // row = query, k-block = key block
      }
      fence_async_smem();  // P^T / dS^T are read by the tensor core
      warp_arrive(BAR(B_PATOM + b), lane);
    }
    // ---- dV (query half 0) and dK (query half 1): TMEM -> bf16
    if (__all_sync(0xFFFFFFFFu, ok) && wwait(BAR(B_KVDONE), 0, abort_flag)) {
      tc_fence_after();
      const uint32_t col = hq == 0 ? COL_DV : COL_DK;
      const float mult = hq == 0 ? 1.0f : a.scale;
      const int64_t tok = sk0 + kpos;
      uint16_t* dst = (hq == 0 ? a.dv : a.dk) + (tok * a.H + h) * 128;
      uint8_t* mxd = hq == 0 ? a.dvmx : a.dkmx;
      uint32_t sfw = 0;  // E8M0 scales of the MXFP8 gradient row, one byte per 32 columns
      // A warp whose 32 key rows all lie inside the sequence sends its rows out
      // by TMA stores of 32-row x 64-column halves staged in shared memory (8 KB
      // per warp in the Q and dO rings, idle now that every GEMM has completed,
      // so both halves are staged without waiting for the first one's store;
      // 128B-swizzled rows): a thread storing its own 256-byte row touches 32
      // rows 2H KB apart per instruction.  Other warps store row by row.
      const bool staged = __all_sync(0xFFFFFFFFu, kvalid);
      const uint32_t stg = base + OFF_Q + uint32_t(warp - 4) * 8192u;
      const CUtensorMap* tmo = hq == 0 ? &a.tm_dv : &a.tm_dk;
      uint32_t vv[64];  // two 32-column loads per wait
#pragma unroll
      for (int c = 0; c < 4; c++) {
        if ((c & 1) == 0) {
          tmem_ld32(tmem + lane_base + col + 32 * c, vv);
          tmem_ld32(tmem + lane_base + col + 32 * c + 32, vv + 32);
          tmem_wait_ld();
          reg_fence32(vv);
          reg_fence32(vv + 32);
        }
        const uint32_t* v = vv + 32 * (c & 1);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; e++) {
          const float x0 = ntile > 0 ? __uint_as_float(v[2 * e]) * mult : 0.0f;
          const float x1 = ntile > 0 ? __uint_as_float(v[2 * e + 1]) * mult : 0.0f;
          __nv_bfloat162 p2 = __floats2bfloat162_rn(x0, x1);
          w[e] = *reinterpret_cast<uint32_t*>(&p2);
        }
        if (staged) {
          const uint32_t half = stg + uint32_t(c >> 1) * 4096u;
#pragma unroll
          for (int v4 = 0; v4 < 4; v4++) {
            const uint32_t chunk = uint32_t((c & 1) * 4 + v4) ^ uint32_t(lane & 7);
            st_shared_v4(half + uint32_t(lane) * 128u + (chunk << 4), w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2],
                         w[4 * v4 + 3]);
          }
          if (c & 1) {
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(tmo, half, 64 * (c >> 1), h, int(tok - lane));
              bulk_commit();
            }
          }
        } else if (kvalid) {
#pragma unroll
          for (int v4 = 0; v4 < 4; v4++)
            *reinterpret_cast<uint4*>(dst + 32 * c + 8 * v4) =
                make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
        }
        if (mxd != nullptr) {
          // the 32 bf16 values of this chunk are one 1x32 block along D,
          // quantized exactly as the ROW quantizer treats a bf16 tensor
          const uint32_t sc = mx_block_e8m0(w);
          sfw |= sc << (8 * c);
          if (kvalid) mx_block_store(mxd + (tok * a.H + h) * 128 + 32 * c, w, sc);
        }
      }
      if (mxd != nullptr) {
        uint8_t* sfc = hq == 0 ? a.dvmx_sfc : a.dkmx_sfc;
        uint8_t* sfp = hq == 0 ? a.dvmx_sfp : a.dkmx_sfp;
        if (kvalid && sfc != nullptr) *reinterpret_cast<uint32_t*>(sfc + (tok * a.H + h) * 4) = sfw;
        // packed ROW atom of this key tile; rows past the sequence hold 0x7F
        if (sfp != nullptr) {
          const int64_t tile = seq_units_before_warp(a.sk, g, 128, lane) + kt;
          *reinterpret_cast<uint32_t*>(sfp + (tile * a.H + h) * 512 + (r & 31) * 16 + (r >> 5) * 4) =
              kvalid ? sfw : 0x7F7F7F7Fu;
        }
      }
      // every store of this warp has completed before the CTA exits
      if (lane == 0) bulk_wait0();
      __syncwarp();
    }
  } else if (warp >= 12) {
    warp_converged();
    // ------------------------------------------------------------ dQ drain
    // dQ^T of each tile: TMEM -> shared staging -> one tiled TMA reduce-add
    // into the global accumulator.
    const int d = (warp & 3) * 32 + lane;
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const bool leader = tid == 12 * 32;
    const int esz = a.dq_mode == 1 ? 2 : 4;
    const uint32_t rowb = 128u * esz;
    // fp32 partials are stored unscaled (the final pass applies the softmax
    // scale); fp16 partials carry scale * static scale to stay in range
    const float mult = a.scale * a.dq_static_scale;
    uint8_t* stg0 = smem + OFF_DQS;
    for (int jj = 0; jj < ntile; jj++) {
      // free the TMEM accumulator first, so that the next tile's dQ^T GEMMs
      // can start while this one is staged and reduced
      const bool okw = wwait(BAR(B_DQFULL), jj & 1, abort_flag);
      float v[64];
      if (okw) {
        tc_fence_after();
        tmem_ld32(tmem + lane_base + COL_DQ, reinterpret_cast<uint32_t*>(v));
        tmem_ld32(tmem + lane_base + COL_DQ + 32, reinterpret_cast<uint32_t*>(v) + 32);
        tmem_wait_ld();
        reg_fence32(reinterpret_cast<uint32_t*>(v));
        reg_fence32(reinterpret_cast<uint32_t*>(v) + 32);
        tc_fence_before();
        warp_arrive(BAR(B_DQEMPTY), lane);
      }
      // the reduction issued two tiles ago has finished reading this staging
      // buffer; all four warps reach the barrier whatever their wait returned,
      // and leave together if any of them gave up
      if (leader) bulk_wait_read1();
      if (!named_bar_and(1, 128, okw)) break;
      uint8_t* stg = stg0 + (jj & 1) * DQS_BYTES;
      if (esz == 4) {
#pragma unroll
        for (int q = 0; q < 64; q++) reinterpret_cast<float*>(stg + q * rowb)[d] = v[q];
      } else {
#pragma unroll
        for (int q = 0; q < 64; q++) reinterpret_cast<__half*>(stg + q * rowb)[d] = __float2half_rn(v[q] * mult);
      }
      fence_async_smem();
      named_bar_sync(1, 128);
      if (leader) {
        // one tiled reduce-add of the 64 x 128 partial; rows past the sequence
        // hold exact zeros (their dS is zero) and rows past the tensor are clipped
        tma_reduce_add_3d(&a.tm_dqacc, base + OFF_DQS + (jj & 1) * DQS_BYTES, 0, h,
                          int(sq0 + int64_t(first + jj) * QT));
        bulk_commit();
      }
    }
    if (leader) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t st) {
  static std::atomic<unsigned long long> attr{0};
  clear_stale_error();
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(attn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                bwd::SMEM_BYTES);
  });
  if (e != cudaSuccess) return e;
  {
    // the preparation kernel also zeroes the dQ accumulator
    // at least one tile per (head, sequence): tile 0 of the first and last
    // sequences also zeroes the rows outside every sequence
    dim3 pg(unsigned(max(1, (a.sq.seqlen + bwd::QT - 1) / bwd::QT)), unsigned(a.H), unsigned(a.sq.nseq));
    if (pg.x > 0) bwd_prep_kernel<<<pg, 256, 0, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  dim3 grid;
  BwdArgs args = a;
  if (a.sk.cu == nullptr) {
    const int nkt = (a.sk.seqlen + bwd::KT - 1) / bwd::KT;
    const int per = a.H * a.sk.nseq;
    // Non-causal: about two waves of CTAs per head group, so the group's fp32
    // dQ rows (head_group * S * 512 bytes, about 20 MB) stay in L2 instead of
    // every reduce-add reading and writing DRAM (measured 1.8x on B8 H32
    // S4096).  Causal: one group of all heads (key tile major), which keeps
    // concurrent CTAs on different heads' dQ rows -- grouping measured 5%
    // slower there, its CTAs' reduce-adds contending for the same rows.
    int sms = sm_count_current_device();
    if (sms <= 0) sms = 148;
    args.head_group = (a.causal || nkt <= 0) ? max(per, 1) : min(per, max(1, (2 * sms + nkt - 1) / nkt));
    grid = dim3(unsigned(nkt * per), 1, 1);
  } else {
    grid = dim3(unsigned((a.sk.seqlen + bwd::KT - 1) / bwd::KT), unsigned(a.H), unsigned(a.sk.nseq));
  }
  if (grid.x > 0 && grid.y > 0 && grid.z > 0) {
    attn_bwd_kernel<<<grid, bwd::NTHREADS, bwd::SMEM_BYTES, st>>>(args);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int64_t n = a.total_q * a.H * 128;
  const float mult = a.dq_mode == 1 ? 1.0f / a.dq_static_scale : a.scale;
  if (a.dqmx == nullptr) {
    bwd_post_kernel<<<unsigned((n + 2047) / 2048), 256, 0, st>>>(a.dq_acc, a.dq, n, a.dq_mode, mult);
  } else {
    bwd_post_mx_kernel<<<unsigned((n / 32 + 255) / 256), 256, 0, st>>>(a.dq_acc, a.dq, n, a.dq_mode, mult,
                                                                       a.dqmx, a.dqmx_sfc);
    if (a.dqmx_sfp != nullptr) {
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      PackArgs p;
      p.sf_compact = a.dqmx_sfc;
      p.tokens = a.total_q;
      p.H = a.H;
      p.D = 128;
      p.mode = 0;
      p.seq = a.sq;
      p.packed_tiles = a.ptiles_q;
      p.sf_packed = a.dqmx_sfp;
      return launch_sf_pack(p, st);
    }
  }
  return cudaGetLastError();
}

unsigned read_status_bwd(cudaStream_t st) {
  unsigned v = 0, z = 0;
  cudaMemcpyFromSymbolAsync(&v, g_status_bwd, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
  cudaMemcpyToSymbolAsync(g_status_bwd, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
  cudaStreamSynchronize(st);
  return v;
}

}  // namespace mxfa
