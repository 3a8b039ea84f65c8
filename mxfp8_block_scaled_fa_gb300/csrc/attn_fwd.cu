// attn_fwd.cu -- MXFP8 block-scaled FlashAttention forward for sm_103a.
//
// What it computes ("Meta's MXFP8 FlashAttention-4 kernel, tackling TMEM
// scale-factor constraints, hits up to 1.6x over BF16", paragraphs 1-2;
// "MXFP8 FlashAttention-4 Hits 2.85 Petaflops in Meta's Production Training",
// section "Inside the TMEM Bargain and Zero-Gather Jagged Pipeline"):
//   S = Q K^T as a block-scaled MMA (E4M3 x E4M3, E8M0 scales per 32 of D),
//   FP32 online softmax in base 2, P converted to MXFP8 in registers in
//   32-key blocks whose scale comes from the block maxima of the scores
//   (bit extraction, no log or division), O += P V as a block-scaled MMA with
//   P read from tensor memory and V scaled per 32 keys.
//
// Structure (one CTA = one 128-query tile of one head, 1 CTA per SM):
//   warp 0      TMA producer: Q once; K, V tiles + their scale atoms into a
//               3-stage shared-memory ring (mbarrier complete_tx)
//   warp 1      TMEM owner and MMA issuer: scale atoms enter TMEM through
//               tcgen05.cp (in issue order with the MMAs); S(j) into one of
//               two TMEM S buffers, then O += P(j-1) V(j-1)
//   warps 4..7  softmax: thread i owns query row i (TMEM lane i); writes
//               P(j) over the first 32 columns of S(j) and its scales to a
//               shared atom; rescales O in TMEM when the running max moves;
//               final O / l and LSE
// TMEM columns: S0 [0,128) S1 [128,256) O [256,384) scales [384,..).
// The running max moves only when it grows by more than kRescaleThr (log2
// units); P~ then stays below 2^kRescaleThr, which the E8M0 block scale
// absorbs, and O and l carry the stale max exactly.
#include <cuda_bf16.h>

#include "mx_ptx.cuh"
#include "mx_seq.cuh"
#include "mxfa_internal.h"

namespace mxfa {

static __device__ unsigned g_status_fwd;

namespace fwd {
constexpr int NS = 3;  // K/V pipeline stages
constexpr int TILE = 128;
constexpr int TILE_BYTES = TILE * 128;  // 128 rows x 128 E4M3
constexpr float kRescaleThr = 8.0f;

constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE_BYTES;
constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
constexpr int OFF_SF = OFF_V + NS * TILE_BYTES;
constexpr int OFF_SFQ = OFF_SF;
constexpr int OFF_SFK = OFF_SFQ + 512;
constexpr int OFF_SFV = OFF_SFK + NS * 512;
constexpr int OFF_SFP = OFF_SFV + NS * 512;
constexpr int NWG = 2;               // softmax warpgroups sharing each S tile
constexpr int W = 128 / NWG;         // key columns per warpgroup
constexpr int NB = W / 32;           // P blocks per thread
constexpr int OFF_RED = OFF_SFP + 2 * 512;             // row maxima [2][NWG][128], sums [NWG][128]
constexpr int OFF_VOTE = OFF_RED + 3 * NWG * 128 * 4;  // exit votes [3][NWG*4]
constexpr int OFF_BAR = OFF_VOTE + 3 * NWG * 4 * 4;
// barriers: q_full, kv_full[NS], kv_empty[NS], s_full[2], p_full[2], o_done, teardown
constexpr int NBAR = 1 + 2 * NS + 2 + 2 + 1 + 1;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack

constexpr uint32_t COL_S0 = 0, COL_O = 256, COL_SFQ = 384, COL_SFK = 388, COL_SFV = 396,
                   COL_SFP = 404;
constexpr int NTHREADS = 128 + NWG * 128;
}  // namespace fwd

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool mbar_wait_raw(uint32_t bar, uint32_t parity) {
  unsigned long long t0 = global_ns();
  while (!mbar_try_wait_sleep(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

__global__ void __launch_bounds__(fwd::NTHREADS, 1) attn_fwd_kernel(const __grid_constant__ FwdArgs a) {
  using namespace fwd;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- work item
  int g, h, qt;
  if (a.sq.cu == nullptr) {  // dense: heavy (late) query tiles first
    const int nqt = (a.sq.seqlen + TILE - 1) / TILE;
    const int per = a.H * a.sq.nseq;
    qt = nqt - 1 - int(blockIdx.x) / per;
    const int bh = int(blockIdx.x) % per;
    g = bh / a.H;
    h = bh % a.H;
  } else {
    qt = blockIdx.x;
    h = blockIdx.y;
    g = blockIdx.z;
  }
  int64_t sq0, sk0;
  int lq, lk;
  seq_info(a.sq, g, sq0, lq);
  seq_info(a.sk, g, sk0, lk);
  if (qt * TILE >= lq) return;  // empty tile of a short sequence (before any setup)
  int nkv = (lk + TILE - 1) / TILE;
  if (a.causal) nkv = min(nkv, qt + 1);
  const int64_t tq_g = seq_units_before(a.sq, g, TILE) + qt;
  const int64_t tk_g0 = seq_units_before(a.sk, g, TILE);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  const uint32_t bar0 = smem_u32(bars);
  auto BAR = [&](int i) { return bar0 + 8u * uint32_t(i); };
  const int B_QFULL = 0, B_KVFULL = 1, B_KVEMPTY = 1 + NS, B_SFULL = 1 + 2 * NS,
            B_PFULL = 3 + 2 * NS, B_ODONE = 5 + 2 * NS, B_TEAR = 6 + 2 * NS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 8);

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(BAR(B_QFULL), 1);
    for (int s = 0; s < NS; s++) {
      mbar_init(BAR(B_KVFULL + s), 1);
      mbar_init(BAR(B_KVEMPTY + s), 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(BAR(B_SFULL + b), 1);
      mbar_init(BAR(B_PFULL + b), NWG * 128);
    }
    mbar_init(BAR(B_ODONE), 1);
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
  const bool bad_tiles = (tq_g >= a.ptiles_q) || (tk_g0 + nkv > a.ptiles_k);
  if (bad_tiles && tid == 0) {
    atomicOr(&g_status_fwd, DEV_BAD_INDEX);
    *abort_flag = 1;
  }
  __syncthreads();

  if (warp == 0 && !bad_tiles) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&a.tm_q);
      tma_prefetch_desc(&a.tm_k);
      tma_prefetch_desc(&a.tm_v);
      mbar_arrive_expect_tx(BAR(B_QFULL), TILE_BYTES + 512);
      tma_load_3d(base + OFF_Q, &a.tm_q, BAR(B_QFULL), 0, h, int(sq0 + int64_t(qt) * TILE));
      bulk_load(base + OFF_SFQ, a.sfq + (tq_g * a.H + h) * 512, 512, BAR(B_QFULL));
      int issued = 0;
      for (int j = 0; j < nkv; j++) {
        const int s = j % NS, u = j / NS;
        if (j >= NS && !mbar_wait(BAR(B_KVEMPTY + s), (u - 1) & 1, abort_flag, &g_status_fwd)) break;
        issued = j + 1;
        const uint32_t fb = BAR(B_KVFULL + s);
        mbar_arrive_expect_tx(fb, 2 * TILE_BYTES + 1024);
        const int krow = int(sk0 + int64_t(j) * TILE);
        tma_load_3d(base + OFF_K + s * TILE_BYTES, &a.tm_k, fb, 0, h, krow);
        tma_load_3d(base + OFF_V + s * TILE_BYTES, &a.tm_v, fb, 0, h, krow);
        const int64_t atom = ((tk_g0 + j) * a.H + h) * 512;
        bulk_load(base + OFF_SFK + s * 512, a.sfk + atom, 512, fb);
        bulk_load(base + OFF_SFV + s * 512, a.sfv + atom, 512, fb);
      }
      // every issued copy has landed before the CTA may exit
      for (int j = max(0, issued - NS); j < issued; j++) mbar_wait_raw(BAR(B_KVFULL + j % NS), (j / NS) & 1);
      mbar_wait_raw(BAR(B_QFULL), 0);
    }
  } else if (warp == 1 && !bad_tiles) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the schedule so that descriptors and TMEM addresses
    // are warp-uniform values; lane 0 alone issues the tcgen05 operations.
    {
      const bool issuer = lane == 0;
      const uint32_t tm = __shfl_sync(0xFFFFFFFFu, tmem, 0);
      auto wait_all = [&](uint32_t bar, uint32_t par) {
        return __all_sync(0xFFFFFFFFu, mbar_wait(bar, par, abort_flag, &g_status_fwd));
      };
      auto cp_sf = [&](uint32_t col, uint32_t saddr) {
        const uint64_t d = smem_desc(saddr, 128, 128, 0);
        if (issuer)
          asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tm + col), "l"(d) : "memory");
      };
      const uint64_t dQ = smem_desc(base + OFF_Q, 16, 1024, 2);
      auto issue_pv = [&](int jj) -> bool {
        const int s = jj % NS, b = jj & 1;
        if (!wait_all(BAR(B_PFULL + b), (jj >> 1) & 1)) return false;
        tc_fence_after();
        cp_sf(COL_SFP + 4 * b, base + OFF_SFP + b * 512);
        cp_sf(COL_SFV + 4 * b, base + OFF_SFV + s * 512);
        const uint64_t dV = smem_desc(base + OFF_V + s * TILE_BYTES, 8192, 1024, 2);
        if (issuer) {
#pragma unroll
          for (int k = 0; k < 4; k++)
            mma_mxf8_ts(tm + COL_O, tm + COL_S0 + 128 * b + 8 * k, dV + uint64_t(256 * k),
                        idesc_mxf8(128, 128, 0, 1, k, k), tm + COL_SFP + 4 * b, tm + COL_SFV + 4 * b,
                        (jj > 0 || k > 0) ? 1u : 0u);
          tc_commit(BAR(B_KVEMPTY + s));
          tc_commit(BAR(B_ODONE));
        }
        __syncwarp();
        return true;
      };
      bool ok = wait_all(BAR(B_QFULL), 0);
      tc_fence_after();
      if (ok) cp_sf(COL_SFQ, base + OFF_SFQ);
      for (int j = 0; ok && j < nkv; j++) {
        const int s = j % NS, b = j & 1;
        if (!wait_all(BAR(B_KVFULL + s), (j / NS) & 1)) { ok = false; break; }
        tc_fence_after();
        cp_sf(COL_SFK + 4 * b, base + OFF_SFK + s * 512);
        const uint64_t dK = smem_desc(base + OFF_K + s * TILE_BYTES, 16, 1024, 2);
        if (issuer) {
#pragma unroll
          for (int k = 0; k < 4; k++)
            mma_mxf8_ss(tm + COL_S0 + 128 * b, dQ + uint64_t(2 * k), dK + uint64_t(2 * k),
                        idesc_mxf8(128, 128, 0, 0, k, k), tm + COL_SFQ, tm + COL_SFK + 4 * b,
                        k > 0 ? 1u : 0u);
          tc_commit(BAR(B_SFULL + b));
        }
        __syncwarp();
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && nkv > 0) issue_pv(nkv - 1);
      // all MMAs of this CTA retired before TMEM is released
      if (issuer) {
        tc_commit(BAR(B_TEAR));
        mbar_wait_raw(BAR(B_TEAR), 0);
      }
      __syncwarp();
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    // NWG warpgroups share each 128 x 128 S tile: warpgroup g owns key columns
    // [g*W, (g+1)*W) of every row (thread = query row = TMEM lane).  They
    // exchange their partial row maxima once per tile; each keeps its own
    // partial row sum, writes its own P columns and rescales its own O columns.
    // Every exit decision is a vote read after a barrier all of them reach, so
    // they always leave together.
    const int gw = (warp - 4) >> 2;
    const int wi = warp - 4;                       // softmax warp index
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const int qpos = qt * TILE + row;
    const float sl2 = a.scale_log2;
    const int c0 = gw * W;
    float* red = reinterpret_cast<float*>(smem + OFF_RED);            // [2][NWG][128]
    volatile int* vote = reinterpret_cast<volatile int*>(smem + OFF_VOTE);  // [2][NWG*4]
    float m = -INFINITY, l = 0.0f;
    bool failed = false, ok = true;
    for (int j = 0; j < nkv; j++) {
      const int b = j & 1;
      const bool okw = !failed &&
          __all_sync(0xFFFFFFFFu, mbar_wait(BAR(B_SFULL + b), (j >> 1) & 1, abort_flag, &g_status_fwd));
      float s[W];
      float bm[NB];
      float pm = -INFINITY;
      const int kbase = j * TILE + c0;
      const int klim = a.causal ? min(lk, qpos + 1) : lk;  // keys < klim are visible
      if (okw) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < W / 32; c++)
          tmem_ld32(tmem + lane_base + COL_S0 + 128 * b + c0 + 32 * c, reinterpret_cast<uint32_t*>(s) + 32 * c);
        tmem_wait_ld();
        const bool need_mask = (kbase + W > lk) || (a.causal && kbase + W - 1 > qpos);
        if (need_mask) {
#pragma unroll
          for (int i = 0; i < W; i++)
            if (kbase + i >= klim) s[i] = -INFINITY;
        }
#pragma unroll
        for (int kb = 0; kb < NB; kb++) {
          float x = s[32 * kb];
#pragma unroll
          for (int i = 1; i < 31; i += 2)
            asm("max.f32 %0, %1, %2, %3;" : "=f"(x) : "f"(x), "f"(s[32 * kb + i]), "f"(s[32 * kb + i + 1]));
          bm[kb] = fmaxf(x, s[32 * kb + 31]);
          pm = fmaxf(pm, bm[kb]);
        }
      }
      red[(b * NWG + gw) * 128 + row] = pm;
      if (lane == 0) vote[b * (NWG * 4) + wi] = okw ? 1 : 0;
      named_bar_sync(2, NWG * 128);
      bool all_ok = true;
#pragma unroll
      for (int v = 0; v < NWG * 4; v++) all_ok = all_ok && vote[b * (NWG * 4) + v] != 0;
      if (!all_ok) { ok = false; break; }
      // raw-score maxima; fl(max S * sl2) = max fl(S * sl2) since sl2 > 0
      float mt = red[(b * NWG + 0) * 128 + row];
#pragma unroll
      for (int g2 = 1; g2 < NWG; g2++) mt = fmaxf(mt, red[(b * NWG + g2) * 128 + row]);
      mt = __fmul_rn(mt, sl2);
      const float mn = fmaxf(m, mt);
      const float mu = (m == -INFINITY || __fsub_rn(mn, m) > kRescaleThr) ? mn : m;
      const float mref = mu == -INFINITY ? 0.0f : mu;
      const float alpha = ex2(__fsub_rn(m, mref));
      const bool rescale = (m != -INFINITY) && (mu > m);
      // P -> E4M3, one E8M0 scale per 32 keys.  The block maximum of P~ is
      // 2^(fl(block max S * sl2) - m) (no second pass over the elements); with
      // its exponent X, each element is put on the E4M3 scale directly as
      // 2^fma(S, sl2, -fl(m + X)) and converted, and the row sum adds
      // 2^X * (block sum).
      uint32_t pw[W / 4];
      uint32_t sfw = 0;
      float lt = 0.0f;
#pragma unroll
      for (int kb = 0; kb < NB; kb++) {
        const uint32_t sc = e8m0_from_amax(ex2(__fsub_rn(__fmul_rn(bm[kb], sl2), mref)));
        sfw |= sc << (8 * kb);
        const float nmx = -__fadd_rn(mref, float(int(sc) - 127));
        float2 rs = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int c = 0; c < 8; c++) {
          float* p = s + 32 * kb + 4 * c;
          const float2 a01 = ffma2(make_float2(p[0], p[1]), make_float2(sl2, sl2), make_float2(nmx, nmx));
          const float2 a23 = ffma2(make_float2(p[2], p[3]), make_float2(sl2, sl2), make_float2(nmx, nmx));
          const float2 x01 = make_float2(ex2(a01.x), ex2(a01.y));
          const float2 x23 = make_float2(ex2(a23.x), ex2(a23.y));
          rs = fadd2(rs, fadd2(x01, x23));
          pw[8 * kb + c] = cvt_e4m3x2(x01.x, x01.y) | (cvt_e4m3x2(x23.x, x23.y) << 16);
        }
        lt += (rs.x + rs.y) * e8m0_value(sc);
      }
      l = l * alpha + lt;
      // O must hold PV(j-1) before it is rescaled and before PV(j) is issued
      if (j >= 1 &&
          !__all_sync(0xFFFFFFFFu, mbar_wait(BAR(B_ODONE), (j - 1) & 1, abort_flag, &g_status_fwd))) {
        failed = true;  // leave at the next vote, together with the others
        m = mu;
        continue;
      }
      tc_fence_after();
      if (__any_sync(0xFFFFFFFFu, rescale)) {
#pragma unroll
        for (int c = 0; c < W / 32; c++) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_base + COL_O + c0 + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 t = fmul2(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                   make_float2(alpha, alpha));
            o[i] = __float_as_uint(t.x);
            o[i + 1] = __float_as_uint(t.y);
          }
          tmem_st16(tmem + lane_base + COL_O + c0 + 32 * c, o);
          tmem_st16(tmem + lane_base + COL_O + c0 + 32 * c + 16, o + 16);
        }
      }
#pragma unroll
      for (int c = 0; c < W / 4; c += 16)
        tmem_st16(tmem + lane_base + COL_S0 + 128 * b + c0 / 4 + c, pw + c);
      uint8_t* atom = smem + OFF_SFP + b * 512 + (row & 31) * 16 + (row >> 5) * 4 + gw * NB;
#pragma unroll
      for (int kb = 0; kb < NB; kb++) atom[kb] = uint8_t(sfw >> (8 * kb));
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(BAR(B_PFULL + b));
      m = mu;
    }
    // ---- epilogue: O / l -> bf16 (each warpgroup its own columns), LSE
    const bool okf = ok && !failed && nkv > 0 &&
        __all_sync(0xFFFFFFFFu, mbar_wait(BAR(B_ODONE), (nkv - 1) & 1, abort_flag, &g_status_fwd));
    float* lsum = red + 2 * NWG * 128;  // [NWG][128]
    lsum[gw * 128 + row] = l;
    if (lane == 0) vote[2 * (NWG * 4) + wi] = okf ? 1 : 0;
    named_bar_sync(2, NWG * 128);
    bool all_ok = true;
#pragma unroll
    for (int v = 0; v < NWG * 4; v++) all_ok = all_ok && vote[2 * (NWG * 4) + v] != 0;
    if (all_ok) {
      tc_fence_after();
      float lt = lsum[row];
#pragma unroll
      for (int g2 = 1; g2 < NWG; g2++) lt += lsum[g2 * 128 + row];
      const bool valid = qpos < lq;
      const float rl = 1.0f / lt;
      uint16_t* orow = a.o + ((sq0 + qpos) * a.H + h) * 128 + c0;
#pragma unroll
      for (int c = 0; c < W / 32; c++) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + COL_O + c0 + 32 * c, o);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int v4 = 0; v4 < 4; v4++) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
              __nv_bfloat162 p2 = __floats2bfloat162_rn(__uint_as_float(o[8 * v4 + 2 * e]) * rl,
                                                        __uint_as_float(o[8 * v4 + 2 * e + 1]) * rl);
              w4[e] = *reinterpret_cast<uint32_t*>(&p2);
            }
            *reinterpret_cast<uint4*>(orow + 32 * c + 8 * v4) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
      if (valid && gw == 0) {
        const float lse = (m + log2f(lt)) * 0.69314718055994530942f;
        if (a.dense_lse)
          a.lse[(int64_t(g) * a.H + h) * a.lse_hstride + qpos] = lse;
        else
          a.lse[int64_t(h) * a.lse_hstride + sq0 + qpos] = lse;
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

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         fwd::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid;
  if (a.sq.cu == nullptr) {
    const int nqt = (a.sq.seqlen + fwd::TILE - 1) / fwd::TILE;
    grid = dim3(unsigned(nqt * a.H * a.sq.nseq), 1, 1);
  } else {
    grid = dim3(unsigned((a.sq.seqlen + fwd::TILE - 1) / fwd::TILE), unsigned(a.H), unsigned(a.sq.nseq));
  }
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  attn_fwd_kernel<<<grid, fwd::NTHREADS, fwd::SMEM_BYTES, st>>>(a);
  return cudaPeekAtLastError();
}

unsigned read_status_fwd(cudaStream_t st) {
  unsigned v = 0, z = 0;
  cudaMemcpyFromSymbolAsync(&v, g_status_fwd, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
  cudaMemcpyToSymbolAsync(g_status_fwd, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
  cudaStreamSynchronize(st);
  return v;
}

}  // namespace mxfa
