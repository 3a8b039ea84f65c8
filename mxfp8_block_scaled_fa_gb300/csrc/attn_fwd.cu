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
// Structure: a persistent kernel, one CTA per SM, 12 warps.  A work item is
// two 128-query tiles (A and B) of one head; each CTA takes item blockIdx.x,
// then claims further items from a global counter in a fixed order (dense:
// late query pairs first, the heavy ones under a causal mask; varlen:
// sequence by sequence), so that the SMs finish together.  The tensor core
// alternates between the tiles, so that one tile's softmax runs while the
// other tile's GEMMs execute:
//   S_A(j), PV_B(j-1), S_B(j), PV_A(j), S_A(j+1), ...
// and the next item's Q and first K/V tiles load while the current one runs
// (Q double-buffered, K/V ring shared by consecutive items).
//   warp 0      TMA producer (lane 0): claims items, publishes them to the
//               other roles through a two-entry ring, loads Q_A, Q_B per item
//               and the K, V tiles + scale atoms through the ring
//   warp 1      TMEM owner and MMA issuer; scale atoms enter TMEM through
//               tcgen05.cp in issue order with the MMAs that read them
//   warps 4-7   softmax of tile A, warps 8-11 softmax of tile B: thread =
//               query row = TMEM lane, the whole 128-key row in registers;
//               the same warps write the item's O and lse
// TMEM (all 512 columns): S_A [0,128) S_B [128,256) O_A [256,384)
// O_B [384,512).  Once a tile's softmax has loaded S_X(j), the columns of S_X
// carry P_X(j) [0,32), its scales [32,36) (both stored by the softmax
// warps), the V scales [36,40) (read by
// PV_X(j)), and the Q / K scales of the other tile's next S GEMM [40,48).
// The running max moves only when it grows by more than a threshold (log2
// units, 8 by default, 0 = at every increase); P~ then stays below
// 2^threshold, which the E8M0 block scale absorbs, and O and l carry the
// stale max exactly.  P's block scales come from the block maxima, or, in the
// constant-scale mode, are one fixed E8M0 byte for every block (the pages'
// constant scaling of softmax outputs, which lie in a known range).  The epilogue writes O as
// bf16 and, on request, also as MXFP8 (the bf16 row quantized in 1x32 blocks
// along D, with compact and packed scales).
#include <cuda_bf16.h>

#include "mx_ptx.cuh"
#include "mx_seq.cuh"
#include "mxfa_internal.h"

namespace mxfa {

static __device__ unsigned g_status_fwd;

// Dynamic work claiming: per launch slot, the next item to hand out (after
// the first gridDim.x, which CTA b takes as item b) and the CTAs finished.
// The last CTA of a launch resets its slot; launches in flight at the same
// time (other streams) use other slots.
constexpr int kFwdSchedSlots = 64;
static __device__ unsigned g_fwd_sched[kFwdSchedSlots][2];

namespace fwd {
constexpr int TILE = 128;
constexpr int TILE_BYTES = TILE * 128;  // 128 rows x 128 E4M3
constexpr int NS_MAX = 4;               // K/V pipeline stages at most

// Q_A, Q_B of two work items (slot = item parity), so that the next item's Q
// lands while this item runs
constexpr int OFF_Q = 0;                               // [slot][tile]
constexpr int OFF_K = OFF_Q + 4 * TILE_BYTES;          // NS stages
enum {
  B_QFULL = 0, B_QEMPTY = B_QFULL + 2, B_SFULL = B_QEMPTY + 2, B_SLOAD = B_SFULL + 2, B_PFULL = B_SLOAD + 2,
  B_ODONE = B_PFULL + 2, B_TEAR = B_ODONE + 2, B_IFULL = B_TEAR + 1, B_IEMPTY = B_IFULL + 2,
  B_KVFULL = B_IEMPTY + 2, B_KVEMPTY = B_KVFULL + NS_MAX, NBAR = B_KVEMPTY + NS_MAX
};
// item ring (2 entries): the producer publishes each claimed item, the MMA
// warp and the eight softmax warps release it
constexpr int ITEM_READERS = 9;
// O staging for TMA stores: one area of 32 rows x 64 bf16 columns (128B-swizzled)
// per softmax warp
constexpr int OST_BYTES = 32 * 128;

// Shared-memory layout.  STAGE: O leaves through TMA stores staged in shared
// memory, paid for with one K/V stage (for short items, where the epilogue is
// a large share of the work); otherwise every thread stores its own O row.
template <bool STAGE>
struct Layout {
  static constexpr int NS = STAGE ? 3 : 4;                 // K/V pipeline stages
  static constexpr int OFF_V = OFF_K + NS * TILE_BYTES;    // NS stages
  static constexpr int OFF_OST = OFF_V + NS * TILE_BYTES;  // 8 staging areas (STAGE)
  static constexpr int OFF_SFQ = OFF_OST + (STAGE ? 8 * OST_BYTES : 0);  // 4 atoms [slot][tile]
  static constexpr int OFF_SFK = OFF_SFQ + 4 * 512;        // NS atoms
  static constexpr int OFF_SFV = OFF_SFK + NS * 512;       // NS atoms
  static constexpr int OFF_BAR = OFF_SFV + NS * 512;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_ITEMS = OFF_MISC + 16;          // int[2]: claimed item per ring entry (-1: none left)
  static constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 227 * 1024, "forward tiles exceed the shared memory of one CTA");
  static_assert(OFF_OST % 1024 == 0, "a 128B-swizzled staging area starts on a 1024-byte boundary");
};

constexpr uint32_t COL_S = 0, COL_O = 256;                       // + 128 * tile
constexpr uint32_t SUB_SFP = 32, SUB_SFV = 36, SUB_SFQ = 40, SUB_SFK = 44;  // inside an S region
constexpr int NTHREADS = 384;
// registers per thread after the split: warps 0-3 give up, the softmax warps take
constexpr int REG_SMALL = 56, REG_SOFTMAX = 224;
static_assert(4 * 32 * REG_SMALL + 8 * 32 * REG_SOFTMAX <= NTHREADS * 168,
              "register split exceeds the launch allocation");
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

// One arrival for the whole warp, after every lane's prior work (each lane
// fences its own tcgen05 / shared-memory writes before calling this).
__device__ __forceinline__ void fwd_warp_arrive(uint32_t bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// ---- work items: (sequence g, head h, query pair qp = queries [256 qp, 256 qp + 256)).
// The item space is every (query pair, sequence, head) up to the longest
// sequence's pair count, late pairs (the heavy ones under a causal mask)
// first; a varlen item whose pair starts past its sequence's end is empty and
// every role skips it.  The count and the item -> (g, h, qp) map use kernel
// parameters only, and the other fields come from loads at warp-uniform
// addresses: the roles' item loops stay warp-uniform, which keeps the MMA
// issuer's tcgen05 code compact and fast.
struct FwdItem {
  int g, h, qp;
  int64_t sq0, sk0;
  int lq, lk;
  bool valid, has_b;
  int nkv_all, nkv_a, nkv_b, nkv_max;  // key tiles in the sequence, for tile A, tile B, either
};

__device__ __forceinline__ int fwd_num_items(const FwdArgs& a) {
  return ((a.sq.seqlen + 2 * fwd::TILE - 1) / (2 * fwd::TILE)) * a.H * a.sq.nseq;
}

__device__ __forceinline__ FwdItem fwd_item(const FwdArgs& a, int item) {
  using namespace fwd;
  FwdItem w;
  const int npair = (a.sq.seqlen + 2 * TILE - 1) / (2 * TILE);
  if (a.sq.cu == nullptr) {  // dense: late (heavy under a causal mask) pairs first
    const int per = a.H * a.sq.nseq;
    w.qp = npair - 1 - item / per;
    const int bh = item % per;
    w.g = bh / a.H;
    w.h = bh % a.H;
  } else {  // varlen: sequence by sequence, each one's late pairs first
    const int per = a.H * npair;
    w.g = item / per;
    const int ph = item % per;
    w.qp = npair - 1 - ph / a.H;
    w.h = ph % a.H;
  }
  seq_info(a.sq, w.g, w.sq0, w.lq);
  seq_info(a.sk, w.g, w.sk0, w.lk);
  w.valid = w.qp * 2 * TILE < w.lq;
  w.has_b = w.qp * 2 * TILE + TILE < w.lq;
  w.nkv_all = (w.lk + TILE - 1) / TILE;
  // key tiles each query tile needs (causal: up to its last query)
  w.nkv_a = a.causal ? min(w.nkv_all, 2 * w.qp + 1) : w.nkv_all;
  w.nkv_b = !w.has_b ? 0 : a.causal ? min(w.nkv_all, 2 * w.qp + 2) : w.nkv_all;
  w.nkv_max = max(w.nkv_a, w.nkv_b);
  return w;
}

// Packed 128-row tiles of the sequences before g (one thread, serial).
__device__ __forceinline__ int64_t tiles_before(const Seqs& s, int g) {
  if (!s.cu) return int64_t(g) * ((s.seqlen + fwd::TILE - 1) / fwd::TILE);
  int64_t acc = 0;
  for (int i = 0; i < g; i++) acc += (__ldg(s.cu + i + 1) - __ldg(s.cu + i) + fwd::TILE - 1) / fwd::TILE;
  return acc;
}

// PCONST: every P block takes the scale a.p_sc_const (the constant-scale mode);
// STAGE: the shared-memory layout with O staging (see Layout)
template <bool PCONST, bool STAGE>
__global__ void __launch_bounds__(fwd::NTHREADS, 1) attn_fwd_kernel(const __grid_constant__ FwdArgs a) {
  using namespace fwd;
  using L = Layout<STAGE>;
  constexpr int NS = L::NS, OFF_V = L::OFF_V, OFF_SFQ = L::OFF_SFQ, OFF_SFK = L::OFF_SFK, OFF_SFV = L::OFF_SFV,
                OFF_BAR = L::OFF_BAR, OFF_MISC = L::OFF_MISC, OFF_ITEMS = L::OFF_ITEMS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- persistent: this CTA takes work items blockIdx.x, blockIdx.x + gridDim.x, ...
  // Every role walks the same item sequence; barrier phases run on per-CTA
  // counters across items (Q slot = item parity; K/V stage and S/P steps on
  // running tile counters).
  const uint32_t bar0 = base + OFF_BAR;
  auto BAR = [&](int i) { return bar0 + 8u * uint32_t(i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 8);
  const int nitems = fwd_num_items(a);

  if (tid == 0) {
    *abort_flag = 0;
    for (int q = 0; q < 2; q++) {
      mbar_init(BAR(B_QFULL + q), 1);
      mbar_init(BAR(B_QEMPTY + q), 1);
    }
    for (int s = 0; s < NS; s++) {
      mbar_init(BAR(B_KVFULL + s), 1);
      mbar_init(BAR(B_KVEMPTY + s), 1);
    }
    for (int x = 0; x < 2; x++) {
      mbar_init(BAR(B_SFULL + x), 1);
      mbar_init(BAR(B_SLOAD + x), 4);  // one arrival per softmax warp
      mbar_init(BAR(B_PFULL + x), 4);
      mbar_init(BAR(B_ODONE + x), 1);
    }
    mbar_init(BAR(B_TEAR), 1);
    for (int r = 0; r < 2; r++) {
      mbar_init(BAR(B_IFULL + r), 1);
      mbar_init(BAR(B_IEMPTY + r), ITEM_READERS);
    }
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
  volatile int* s_items = reinterpret_cast<volatile int*>(smem + OFF_ITEMS);
  // ring entry r (whole warp): wait until published, read it, release it
  auto take_item = [&](int r, bool& ok) {
    ok = ok && __all_sync(0xFFFFFFFFu, mbar_wait(BAR(B_IFULL + (r & 1)), (r >> 1) & 1, abort_flag, &g_status_fwd));
    const int it = ok ? s_items[r & 1] : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(BAR(B_IEMPTY + (r & 1)));
    return it;
  };
  // register split (whole warpgroups): the softmax rows live in registers
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REG_SMALL));
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      // Lane 0 alone walks the items, waits for free slots and issues the
      // copies.
      if (lane == 0) {
        tma_prefetch_desc(&a.tm_q);
        tma_prefetch_desc(&a.tm_k);
        tma_prefetch_desc(&a.tm_v);
        int kv = 0;  // key tiles loaded
        int k = 0;   // non-empty items whose Q was loaded (slot = item parity)
        bool ok = true;
        for (int r = 0;; r++) {
          // claim the next item and publish it in ring entry r & 1, once
          // every reader has released entry r - 2
          if (r >= 2 && !mbar_wait(BAR(B_IEMPTY + (r & 1)), ((r >> 1) - 1) & 1, abort_flag, &g_status_fwd)) break;
          int it = r == 0 ? int(blockIdx.x) : int(gridDim.x + atomicAdd(&g_fwd_sched[a.sched_slot][0], 1u));
          FwdItem w = fwd_item(a, ok && it < nitems ? it : 0);
          // a varlen item whose query pair lies past its sequence is skipped
          // here rather than passed through the ring to every reader (dense
          // items are never empty)
          while (a.sq.cu != nullptr && ok && it < nitems && !w.valid) {
            it = int(gridDim.x + atomicAdd(&g_fwd_sched[a.sched_slot][0], 1u));
            if (it < nitems) w = fwd_item(a, it);
          }
          if (!ok || it >= nitems) it = -1;
          s_items[r & 1] = it;
          mbar_arrive(BAR(B_IFULL + (r & 1)));
          if (it < 0) break;
          if (!w.valid) continue;
          const int64_t tq_g = tiles_before(a.sq, w.g) + 2 * w.qp;  // packed tile of Q_A
          const int64_t tk_g0 = tiles_before(a.sk, w.g);            // packed tile of key tile 0
          // an item whose packed tiles fall outside the caller's buffers stops the run
          if (tq_g + (w.has_b ? 2 : 1) > a.ptiles_q || tk_g0 + w.nkv_all > a.ptiles_k) {
            atomicOr(&g_status_fwd, DEV_BAD_INDEX);
            *abort_flag = 1;
            break;
          }
          const int qs = k & 1;
          // slot qs held the Q of item k - 2, released after its last GEMM
          if (k >= 2 && !mbar_wait(BAR(B_QEMPTY + qs), ((k >> 1) - 1) & 1, abort_flag, &g_status_fwd)) break;
          mbar_arrive_expect_tx(BAR(B_QFULL + qs), (w.has_b ? 2 : 1) * (TILE_BYTES + 512));
          const int qrow = int(w.sq0 + int64_t(w.qp) * 2 * TILE);
          tma_load_3d(base + OFF_Q + (2 * qs) * TILE_BYTES, &a.tm_q, BAR(B_QFULL + qs), 0, w.h, qrow);
          bulk_load(base + OFF_SFQ + (2 * qs) * 512, a.sfq + (tq_g * a.H + w.h) * 512, 512, BAR(B_QFULL + qs));
          if (w.has_b) {
            tma_load_3d(base + OFF_Q + (2 * qs + 1) * TILE_BYTES, &a.tm_q, BAR(B_QFULL + qs), 0, w.h,
                        qrow + TILE);
            bulk_load(base + OFF_SFQ + (2 * qs + 1) * 512, a.sfq + ((tq_g + 1) * a.H + w.h) * 512, 512,
                      BAR(B_QFULL + qs));
          }
          k++;
          for (int j = 0; j < w.nkv_max; j++, kv++) {
            const int s = kv % NS, u = kv / NS;
            if (kv >= NS && !mbar_wait(BAR(B_KVEMPTY + s), (u - 1) & 1, abort_flag, &g_status_fwd)) {
              ok = false;
              break;
            }
            const uint32_t fb = BAR(B_KVFULL + s);
            mbar_arrive_expect_tx(fb, 2 * TILE_BYTES + 1024);
            const int krow = int(w.sk0 + int64_t(j) * TILE);
            tma_load_3d(base + OFF_K + s * TILE_BYTES, &a.tm_k, fb, 0, w.h, krow);
            tma_load_3d(base + OFF_V + s * TILE_BYTES, &a.tm_v, fb, 0, w.h, krow);
            const int64_t atom = ((tk_g0 + j) * a.H + w.h) * 512;
            bulk_load(base + OFF_SFK + s * 512, a.sfk + atom, 512, fb);
            bulk_load(base + OFF_SFV + s * 512, a.sfv + atom, 512, fb);
          }
        }
        // every issued copy has landed before the CTA may exit
        for (int j = max(0, kv - NS); j < kv; j++) mbar_wait_raw(BAR(B_KVFULL + j % NS), (j / NS) & 1);
        for (int q = max(0, k - 2); q < k; q++) mbar_wait_raw(BAR(B_QFULL + (q & 1)), (q >> 1) & 1);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp walks the schedule (descriptors and TMEM addresses are
      // warp-uniform) and issues every tcgen05 operation through a lane elected
      // inside the instruction.
      const uint32_t tm = __shfl_sync(0xFFFFFFFFu, tmem, 0);
      auto wait_all = [&](uint32_t bar, uint32_t par) {
        return __all_sync(0xFFFFFFFFu, mbar_wait(bar, par, abort_flag, &g_status_fwd));
      };
      // scale atom (shared memory) -> TMEM, replicated to the four lane quadrants
      auto cp_sf = [&](uint32_t col, uint32_t saddr) {
        tc_cp_sf_w(tm + col, smem_desc(saddr, 128, 128, 0));
      };
      // S_X = Q_X K^T for key tile kvg (global index) from Q slot qs; its scales
      // go into the other tile's S columns, which that tile's softmax has
      // already loaded (or never used)
      auto issue_s = [&](int x, int qs, int kvg) {
        const int s = kvg % NS;
        const uint32_t other = COL_S + 128u * uint32_t(1 - x);
        cp_sf(other + SUB_SFQ, base + OFF_SFQ + 512 * (2 * qs + x));
        cp_sf(other + SUB_SFK, base + OFF_SFK + s * 512);
        const uint64_t dQ = smem_desc(base + OFF_Q + (2 * qs + x) * TILE_BYTES, 16, 1024, 2);
        const uint64_t dK = smem_desc(base + OFF_K + s * TILE_BYTES, 16, 1024, 2);
#pragma unroll
        for (int k = 0; k < 4; k++)
          mma_mxf8_ss_w(tm + COL_S + 128 * x, dQ + uint64_t(2 * k), dK + uint64_t(2 * k),
                        idesc_mxf8(128, 128, 0, 0, k, k), tm + other + SUB_SFQ, tm + other + SUB_SFK,
                        k > 0 ? 1u : 0u);
        tc_commit_w(BAR(B_SFULL + x));
      };
      // O_X (+)= P_X V for key tile kvg, P_X read from the S_X columns (P_X
      // written); the item's first PV starts the accumulator afresh
      auto issue_pv = [&](int x, int kvg, bool first, bool release) {
        const int s = kvg % NS;
        const uint32_t sx = COL_S + 128u * uint32_t(x);
        cp_sf(sx + SUB_SFV, base + OFF_SFV + s * 512);
        const uint64_t dV = smem_desc(base + OFF_V + s * TILE_BYTES, 8192, 1024, 2);
#pragma unroll
        for (int k = 0; k < 4; k++)
          mma_mxf8_ts_w(tm + COL_O + 128 * x, tm + sx + 8 * k, dV + uint64_t(256 * k),
                        idesc_mxf8(128, 128, 0, 1, k, k), tm + sx + SUB_SFP, tm + sx + SUB_SFV,
                        (!first || k > 0) ? 1u : 0u);
        tc_commit_w(BAR(B_ODONE + x));
        // the last GEMM that reads K / V of the stage releases it
        if (release) tc_commit_w(BAR(B_KVEMPTY + s));
      };
      auto kv_ready = [&](int kvg) { return wait_all(BAR(B_KVFULL + kvg % NS), (kvg / NS) & 1); };
      // Per item: S_A(0), S_B(0), then per key tile j two blocks,
      //   A: PV_A(j), S_A(j+1)   B: PV_B(j), S_B(j+1)
      // each issued back to back once everything both GEMMs wait for is in:
      // P_X(j) written; K/V(j+1) landed; the other tile's S loaded by its
      // softmax (its columns take this tile's S scales).  The item's first S
      // GEMMs follow the previous item's last PV GEMMs in this stream; its
      // first PV GEMMs wait (through P) for the softmax warps, which read the
      // previous item's O before they start on this one.
      int kv = 0, k = 0;    // key tiles passed, non-empty items started
      int sa = 0, sb = 0;   // S GEMMs issued per tile (running step counters)
      bool ok = true, done = false;
      int r = 0;            // item ring entries read
      // The item loop runs a trip count fixed by the kernel's arguments (no
      // CTA takes more than nitems + 1 ring entries) and skips its remaining
      // turns once the run is over: a loop whose exit depended on the claimed
      // items would no longer be warp-uniform to the compiler, and the
      // tcgen05 issue code inside it would grow and slow down several-fold.
      // Two levels keep the skipped turns few.
#pragma unroll 1
      for (int r0 = 0; r0 <= nitems; r0 += 32) {
        if (done) continue;
#pragma unroll 1
      for (int r1 = 0; r1 < 32; r1++) {
        if (done) continue;
        const int it = take_item(r++, ok);
        if (it < 0) {
          done = true;
          continue;
        }
        const FwdItem w = fwd_item(a, it);
        if (!w.valid) continue;
        const int qs = k & 1;
        const int nkv_a = w.nkv_a, nkv_b = w.nkv_b;
        ok = wait_all(BAR(B_QFULL + qs), (k >> 1) & 1) && (w.nkv_max == 0 || kv_ready(kv));
        // One copy of the issue code serves both tiles (x is a runtime value):
        // the issuer's code stays small, which keeps it in the instruction
        // cache between blocks.
#pragma unroll 1
        for (int x = 0; ok && x < 2; x++) {
          if ((x ? nkv_b : nkv_a) == 0) continue;
          // S_B(0)'s scales go into A's columns: A's softmax has loaded S_A(0)
          if (x == 1) ok = nkv_a == 0 || wait_all(BAR(B_SLOAD + 0), sa & 1);
          tc_fence_after();
          if (ok) issue_s(x, qs, kv);
        }
        // blocks (j, x) in issue order, A before B for each key tile j
#pragma unroll 1
        for (int bl = 0; ok && bl < 2 * w.nkv_max; bl++) {
          const int j = bl >> 1, x = bl & 1;
          const int n_x = x ? nkv_b : nkv_a, n_o = x ? nkv_a : nkv_b;
          if (j >= n_x) continue;
          const bool next = j + 1 < n_x;
          // S_X(j+1) takes its scales into the other tile's columns, which must
          // hold a loaded S: S_B(j) for block A, S_A(j+1) for block B.  The
          // waits that usually complete first come first, P_X(j) last.
          const int jo = j + x;
          ok = (!next || jo >= n_o || wait_all(BAR(B_SLOAD + 1 - x), ((x ? sa : sb) + jo) & 1)) &&
               (!next || kv_ready(kv + j + 1)) && wait_all(BAR(B_PFULL + x), ((x ? sb : sa) + j) & 1);
          if (!ok) break;
          tc_fence_after();
          // the last GEMM reading K/V(j) releases it: PV_B(j), or PV_A(j) when
          // B has no tile j
          issue_pv(x, kv + j, j == 0, x == 1 || j >= nkv_b);
          if (next) issue_s(x, qs, kv + j + 1);
        }
        // Q slot qs is free once this item's GEMMs have completed
        tc_commit_w(BAR(B_QEMPTY + qs));
        kv += w.nkv_max;
        sa += nkv_a;
        sb += nkv_b;
        k++;
        if (!ok) done = true;
      }
      }
      // all MMAs of this CTA retired before TMEM is released
      tc_commit_w(BAR(B_TEAR));
      mbar_wait_raw(BAR(B_TEAR), 0);
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REG_SOFTMAX));
    // ------------------------------------------------------------ softmax
    // Warpgroup x owns query tile x of every item: thread = query row = TMEM
    // lane, and the whole 128-key row of S_X(j) is loaded into registers at
    // once, which frees the S_X columns for the other tile's scales right
    // away.  After an item's last step the same warps write its O and lse,
    // then go on to the next item, whose first S GEMM is usually done.
    const int x = (warp - 4) >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t col_s = COL_S + 128u * uint32_t(x), col_o = COL_O + 128u * uint32_t(x);
    const float sl2 = a.scale_log2;
    int st = 0;  // S_X steps of earlier items (running barrier phase)
    bool ok = true;
    for (int r = 0; ok; r++) {
      const int it = take_item(r, ok);
      if (it < 0) break;
      const FwdItem wi = fwd_item(a, it);
      if (!wi.valid) continue;
      const int qpos = wi.qp * 2 * TILE + x * TILE + row;
      const int klim = a.causal ? min(wi.lk, qpos + 1) : wi.lk;  // keys < klim are visible
      const int nkv_x = x == 0 ? wi.nkv_a : wi.nkv_b;
      float m = -INFINITY, l = 0.0f;
      for (int j = 0; ok && j < nkv_x; j++) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(BAR(B_SFULL + x), (st + j) & 1, abort_flag, &g_status_fwd))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[128];
  #pragma unroll
        for (int c = 0; c < 4; c++)
          tmem_ld32(tmem + lane_base + col_s + 32 * c, reinterpret_cast<uint32_t*>(s) + 32 * c);
        tmem_wait_ld();
  #pragma unroll
        for (int c = 0; c < 4; c++) reg_fence32(reinterpret_cast<uint32_t*>(s) + 32 * c);
        tc_fence_before();
        fwd_warp_arrive(BAR(B_SLOAD + x), lane);
        const int kbase = j * TILE;
        if (__any_sync(0xFFFFFFFFu, kbase + TILE > klim)) {
  #pragma unroll
          for (int i = 0; i < 128; i++)
            if (kbase + i >= klim) s[i] = -INFINITY;
        }
        // raw-score block maxima (32 keys each) and row maximum
        float bm[4];
        float pm = -INFINITY;
  #pragma unroll
        for (int kb = 0; kb < 4; kb++) {
          float v = s[32 * kb];
  #pragma unroll
          for (int i = 1; i < 31; i += 2) v = fmax3(v, s[32 * kb + i], s[32 * kb + i + 1]);
          bm[kb] = fmaxf(v, s[32 * kb + 31]);
          pm = fmaxf(pm, bm[kb]);
        }
        // fl(max S * sl2) = max fl(S * sl2) since sl2 > 0
        const float mt = __fmul_rn(pm, sl2);
        const float mn = fmaxf(m, mt);
        const float mu = (m == -INFINITY || __fsub_rn(mn, m) > a.rescale_thr) ? mn : m;
        const float mref = mu == -INFINITY ? 0.0f : mu;
        const float alpha = ex2(__fsub_rn(m, mref));
        const bool rescale = (m != -INFINITY) && (mu > m);
        // P -> E4M3, one E8M0 scale per 32 keys.  The block maximum of P~ is
        // 2^(fl(block max S * sl2) - m) (no second pass over the elements); with
        // its exponent X, each element is put on the E4M3 scale directly as
        // 2^fma(S, sl2, -fl(m + X)) and converted, and the row sum adds
        // 2^X * (block sum).
        uint32_t pw[32];
        uint32_t sfw = 0;
        float lt = 0.0f;
  #pragma unroll
        for (int kb = 0; kb < 4; kb++) {
          const uint32_t sc =
              PCONST ? a.p_sc_const : e8m0_from_amax(ex2(__fsub_rn(__fmul_rn(bm[kb], sl2), mref)));
          sfw |= sc << (8 * kb);
          const float nmx = -__fadd_rn(mref, float(int(sc) - 127));
          float2 rs = make_float2(0.0f, 0.0f);
  #pragma unroll
          for (int c = 0; c < 8; c++) {
            const float* p = s + 32 * kb + 4 * c;
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
        // O_X holds PV_X(j-1): S_X(j) completed, and its commit covers every
        // earlier MMA of the issuer.  PV_X(j) waits for this tile's P.
        if (__any_sync(0xFFFFFFFFu, rescale)) {
  #pragma unroll
          for (int c = 0; c < 4; c++) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + col_o + 32 * c, o);
            tmem_wait_ld();
  #pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 t = fmul2(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                     make_float2(alpha, alpha));
              o[i] = __float_as_uint(t.x);
              o[i + 1] = __float_as_uint(t.y);
            }
            tmem_st16(tmem + lane_base + col_o + 32 * c, o);
            tmem_st16(tmem + lane_base + col_o + 32 * c + 16, o + 16);
          }
        }
        tmem_st16(tmem + lane_base + col_s, pw);
        tmem_st16(tmem + lane_base + col_s + 16, pw + 16);
        // this row's four P scales straight into the P scale slot: the MMA
        // reads the scales of rows 32q..32q+31 from lane quadrant q, column q of
        // the slot (the layout a replicated 32x128b copy produces), which is
        // this thread's own lane
        tmem_st1(tmem + lane_base + col_s + SUB_SFP + uint32_t(row >> 5), sfw);
        tmem_wait_st();
        tc_fence_before();
        fwd_warp_arrive(BAR(B_PFULL + x), lane);
        m = mu;
      }
      // ---- epilogue: O / l -> bf16, LSE.  A tile with no key to visit (an
      // empty key sequence) writes O = 0 and lse = -inf, the empty softmax sum.
      const int g = wi.g, h = wi.h, lq = wi.lq;
      const int64_t sq0 = wi.sq0;
      const bool tile_exists = x == 0 || wi.has_b;
      if (ok && tile_exists &&
          (nkv_x == 0 ||
           __all_sync(0xFFFFFFFFu, mbar_wait(BAR(B_ODONE + x), (st + nkv_x - 1) & 1, abort_flag, &g_status_fwd)))) {
        tc_fence_after();
        const bool valid = qpos < lq;
        const bool any_key = nkv_x > 0;
        const float rl = 1.0f / l;
        const int64_t tok = sq0 + qpos;
        uint16_t* orow = a.o + (tok * a.H + h) * 128;
        uint32_t sfw = 0;  // E8M0 scales of the MXFP8 O row, one byte per 32 columns
        // STAGE: a warp whose 32 rows all lie inside the sequence sends O out
        // by TMA stores of 32-row x 64-column halves staged in shared memory
        // (128B-swizzled rows); one thread per row storing its own 256 bytes
        // touches 32 rows 2H KB apart per instruction, which makes the
        // epilogue about as long as two key-tile steps.  Other warps store
        // row by row.
        const bool staged = STAGE && __all_sync(0xFFFFFFFFu, valid);
        const uint32_t ost = base + L::OFF_OST + uint32_t(warp - 4) * OST_BYTES;
        // the row's 128 accumulator columns, all four loads in flight at once
        uint32_t oa[128];
        if (any_key) {
  #pragma unroll
          for (int c = 0; c < 4; c++) tmem_ld32(tmem + lane_base + col_o + 32 * c, oa + 32 * c);
          tmem_wait_ld();
  #pragma unroll
          for (int c = 0; c < 4; c++) reg_fence32(oa + 32 * c);
        } else {
  #pragma unroll
          for (int e = 0; e < 128; e++) oa[e] = 0u;
        }
  #pragma unroll
        for (int c = 0; c < 4; c++) {
          const uint32_t* o = oa + 32 * c;
          const float r = any_key ? rl : 0.0f;
          uint32_t w[16];
  #pragma unroll
          for (int e = 0; e < 16; e++) {
            __nv_bfloat162 p2 = __floats2bfloat162_rn(__uint_as_float(o[2 * e]) * r,
                                                      __uint_as_float(o[2 * e + 1]) * r);
            w[e] = *reinterpret_cast<uint32_t*>(&p2);
          }
          if (staged) {
            // the previous store from this area has read it
            if ((c & 1) == 0) {
              if (lane == 0) bulk_wait_read0();
              __syncwarp();
            }
  #pragma unroll
            for (int v4 = 0; v4 < 4; v4++) {
              const uint32_t chunk = uint32_t((c & 1) * 4 + v4) ^ uint32_t(lane & 7);
              st_shared_v4(ost + uint32_t(lane) * 128u + (chunk << 4), w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2],
                           w[4 * v4 + 3]);
            }
            if (c & 1) {
              fence_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(&a.tm_o, ost, 64 * (c >> 1), h, int(sq0 + qpos - lane));
                bulk_commit();
              }
            }
          } else if (valid) {
  #pragma unroll
            for (int v4 = 0; v4 < 4; v4++)
              *reinterpret_cast<uint4*>(orow + 32 * c + 8 * v4) =
                  make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
          }
          if (a.omx != nullptr) {
            // O as MXFP8: these 32 bf16 values form one 1x32 block along D,
            // quantized exactly as the ROW quantizer treats a bf16 tensor
            const uint32_t sc = mx_block_e8m0(w);
            sfw |= sc << (8 * c);
            if (valid) mx_block_store(a.omx + (tok * a.H + h) * 128 + 32 * c, w, sc);
          }
        }
        if (a.omx != nullptr) {
          if (valid && a.omx_sfc != nullptr)
            *reinterpret_cast<uint32_t*>(a.omx_sfc + (tok * a.H + h) * 4) = sfw;
          // packed ROW atom of this query tile; rows past the sequence hold 0x7F
          if (a.omx_sfp != nullptr) {
            const int64_t tile = seq_units_before_warp(a.sq, g, TILE, lane) + 2 * wi.qp + x;
            *reinterpret_cast<uint32_t*>(a.omx_sfp + (tile * a.H + h) * 512 + (row & 31) * 16 + (row >> 5) * 4) =
                valid ? sfw : 0x7F7F7F7Fu;
          }
        }
        if (valid) {
          const float lse = any_key ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
          if (a.dense_lse)
            a.lse[(int64_t(g) * a.H + h) * a.lse_hstride + qpos] = lse;
          else
            a.lse[int64_t(h) * a.lse_hstride + sq0 + qpos] = lse;
        }
      }
      st += nkv_x;
    }
    // every O store of this warp has completed before the CTA exits
    if (STAGE && lane == 0) bulk_wait0();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  // this CTA claims no more items; the last CTA to finish resets the slot
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&g_fwd_sched[a.sched_slot][1], 1u) == gridDim.x - 1) {
      atomicExch(&g_fwd_sched[a.sched_slot][0], 0u);
      atomicExch(&g_fwd_sched[a.sched_slot][1], 0u);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t st) {
  static std::atomic<unsigned long long> attr{0};
  clear_stale_error();
  cudaError_t e = once_per_device(attr, [] {
    const cudaFuncAttribute smem = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t r = cudaFuncSetAttribute(attn_fwd_kernel<false, false>, smem, fwd::Layout<false>::SMEM_BYTES);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(attn_fwd_kernel<true, false>, smem, fwd::Layout<false>::SMEM_BYTES);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(attn_fwd_kernel<false, true>, smem, fwd::Layout<true>::SMEM_BYTES);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(attn_fwd_kernel<true, true>, smem, fwd::Layout<true>::SMEM_BYTES);
    return r;
  });
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (fewer when there are fewer items); each CTA
  // walks the work items with stride gridDim.x
  const int nsm = sm_count_current_device();
  if (nsm <= 0) return cudaErrorInvalidDevice;
  if (a.H <= 0 || a.sq.nseq <= 0 || a.sq.seqlen <= 0) return cudaSuccess;
  const int64_t items = int64_t((a.sq.seqlen + 2 * fwd::TILE - 1) / (2 * fwd::TILE)) * a.H * a.sq.nseq;
  // item indices (and the strided walk past the last one) stay within 32 bits
  if (items > int64_t(0x7FFFFFFF) - 65536) return cudaErrorInvalidValue;
  const dim3 grid(unsigned(items < nsm ? items : int64_t(nsm)), 1, 1);
  static std::atomic<unsigned> launches{0};
  FwdArgs b = a;
  b.sched_slot = int(launches.fetch_add(1u) % unsigned(kFwdSchedSlots));
  const int sb = b.stage_o ? fwd::Layout<true>::SMEM_BYTES : fwd::Layout<false>::SMEM_BYTES;
  if (b.p_sc_const && b.stage_o)
    attn_fwd_kernel<true, true><<<grid, fwd::NTHREADS, sb, st>>>(b);
  else if (b.p_sc_const)
    attn_fwd_kernel<true, false><<<grid, fwd::NTHREADS, sb, st>>>(b);
  else if (b.stage_o)
    attn_fwd_kernel<false, true><<<grid, fwd::NTHREADS, sb, st>>>(b);
  else
    attn_fwd_kernel<false, false><<<grid, fwd::NTHREADS, sb, st>>>(b);
  return cudaGetLastError();
}

unsigned read_status_fwd(cudaStream_t st) {
  unsigned v = 0, z = 0;
  cudaMemcpyFromSymbolAsync(&v, g_status_fwd, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
  cudaMemcpyToSymbolAsync(g_status_fwd, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
  cudaStreamSynchronize(st);
  return v;
}

}  // namespace mxfa
