// mx_ptx.cuh -- inline-PTX building blocks for sm_103a: mbarriers with bounded
// waits, TMA tile loads, tcgen05 (TMEM alloc, block-scaled MMA, commit,
// ld/st), and the shared-memory / instruction descriptors of the 5th-gen
// tensor core.  Written from the public PTX ISA description of these
// instructions; no vendor library code.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace mxfa {

// Device-side failure codes recorded in a per-module status word.
enum : unsigned {
  DEV_OK = 0,
  DEV_TIMEOUT = 1,     // a bounded wait gave up
  DEV_BAD_INDEX = 2,   // an index check skipped an access
};

// Wait limit for every spin on an mbarrier: 2 s of global time.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of phase `parity` (acquire semantics when it returns true).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// As mbar_try_wait, but a thread whose phase has not completed may sleep (up
// to the hint, 1 ms) until it does, instead of spinning on the issue slots
// that the working warps need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

// Bounded wait on phase `parity` of an mbarrier.  Returns false (and raises
// *abort and the status word) if the barrier has not completed within the
// wait limit or if another role of the CTA already aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          unsigned* status) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (*abort) return false;
    if ((i & 15u) == 0 && global_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      atomicOr(status, DEV_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Plain bulk copy global -> shared (both 16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Bulk reduce-add shared -> global (fp32 / fp16), tracked by bulk groups.
__device__ __forceinline__ void bulk_reduce_add_f32(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(dst),
               "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_reduce_add_f16(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile(
      "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.noftz.f16 [%0], [%1], %2;" ::"l"(dst),
      "r"(src), "r"(bytes)
      : "memory");
}
// Tiled tensor reduce-add shared -> global (element type from the map).
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* m, uint32_t src, int c0, int c1,
                                                  int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(c0), "r"(c1), "r"(c2), "r"(src)
      : "memory");
}
// Tiled tensor store shared -> global, tracked by bulk groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(c0), "r"(c1), "r"(c2), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// 16-byte shared-memory store at a shared-window address.
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
// Make generic-proxy shared-memory writes visible to the async proxy (MMA/TMA).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// States that the whole warp is converged here: an .aligned instruction
// that waits for nothing (no tcgen05.st of this thread is in flight at the
// start of a warp role).  The compiler cannot see that a branch on the warp
// index keeps warps whole; without this statement at the top of each role,
// the tcgen05 issue code inside is compiled for a possibly diverged warp,
// about four times larger and correspondingly slower to issue.
__device__ __forceinline__ void warp_converged() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrive on an mbarrier once all prior tcgen05 async operations of this
// thread have completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc)^T with E8M0 scales from TMEM.
__device__ __forceinline__ void mma_mxf8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Same with the A operand read from TMEM (K-major, 4 E4M3 per column).
__device__ __forceinline__ void mma_mxf8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Warp-wide forms: the whole (converged) warp executes the instruction and
// one lane elected inside it issues the operation.  An issuing warp that
// shares its SM sub-partition with arithmetic-heavy warps issues tcgen05
// operations markedly faster this way than from a lane-0 branch.
__device__ __forceinline__ void mma_mxf8_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %6, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_mxf8_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %6, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit_w(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}
// 512-byte scale atom (shared memory) -> TMEM columns col..col+3, replicated to
// the four lane quadrants (32x128b x4).
__device__ __forceinline__ void tc_cp_sf_w(uint32_t tmem_col, uint64_t sdesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(tmem_col), "l"(sdesc)
      : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with E4M3 A/B, E8M0 scales,
// fp32 accumulation.  a_mn / b_mn: 1 = operand is MN-major in smem.
// sfa_id / sfb_id select the byte of each 32-bit scale column.
// a_fmt / b_fmt: element format codes of the kind (0 E4M3, 3 E2M3, 4 E3M2,
// 5 E2M1).  The sub-byte formats sit in shared memory as runs of 16 codes
// packed little-endian and padded to 16 bytes (one byte per element).
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, int a_mn, int b_mn, int sfa_id,
                                                  int sfb_id, int a_fmt = 0, int b_fmt = 0) {
  return (uint32_t(sfb_id & 3) << 4)       // B scale-factor id
         | (uint32_t(a_fmt & 7) << 7) | (uint32_t(b_fmt & 7) << 10)  // A, B element formats
         | (uint32_t(a_mn & 1) << 15)      // A major
         | (uint32_t(b_mn & 1) << 16)      // B major
         | (uint32_t(N >> 3) << 17)        // N / 8
         | (1u << 23)                      // scale type E8M0
         | (uint32_t(M >> 4) << 24)        // M / 16
         | (uint32_t(sfa_id & 3) << 29);   // A scale-factor id
}

// Shared-memory matrix descriptor (tcgen05 version).
//   swizzle: 0 none, 2 = 128B, 4 = 64B, 6 = 32B
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFF) >> 4);
  d |= uint64_t((lbo & 0x3FFFF) >> 4) << 16;
  d |= uint64_t((sbo & 0x3FFFF) >> 4) << 32;
  d |= uint64_t(1) << 46;  // descriptor version for tcgen05
  d |= uint64_t(swizzle & 7) << 61;
  return d;
}

// TMEM loads/stores: warp w of a warpgroup reaches lanes 32*(w%4) .. +31;
// one 32-bit column per register.
#define MXFA_TMEM_LD_X(N, ...)                                                              \
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x" #N ".b32 " __VA_ARGS__);

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c,
                                         uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(a),
               "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t a) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(a) : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
               "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Marks the 32 registers as (re)defined here, after a tcgen05.wait::ld, so that
// no use of a tcgen05.ld destination is scheduled before the wait.
__device__ __forceinline__ void reg_fence32(uint32_t* r) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                 "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
                 "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
                 "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
                 "+r"(r[31]));
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// TMEM address of (lane, column).
__device__ __forceinline__ uint32_t taddr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

// Named barrier among `nthreads` threads (multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------ MX arithmetic
// E8M0 scale byte from a non-negative fp32 block maximum by bit extraction:
// exponent field - 8 (largest E4M3 exponent), clamped at 0; non-finite -> 0xFF.
__device__ __forceinline__ uint32_t e8m0_from_amax(float amax) {
  uint32_t e = (__float_as_uint(amax) >> 23) & 0xFFu;
  if (e == 0xFFu) return 0xFFu;
  return e > 8u ? e - 8u : 0u;
}
// 2^(127 - s) as fp32 (the factor that maps a block onto the E4M3 range);
// s <= 253 keeps it a normal number.
__device__ __forceinline__ float e8m0_inv_scale(uint32_t s) {
  return __uint_as_float((254u - s) << 23);
}
// Three-input fp32 maximum / minimum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// Named barrier `id` over `n` threads that also returns the AND of `v` over them.
__device__ __forceinline__ bool named_bar_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(v)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
// Packed fp32 pair multiply (one f32x2 instruction), round to nearest.
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(r)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&r);
}
// Packed fp32 pair fused multiply-add a * b + c (one rounding per element).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(r)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
        "l"(*reinterpret_cast<const uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&r);
}
// Packed fp32 pair add.
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(r)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&r);
}
// 2^(s - 127) for an E8M0 byte s in [0, 254] as fp32 (2^-127 is subnormal).
__device__ __forceinline__ float e8m0_value(uint32_t s) {
  return s == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(s << 23);
}
// Two fp32 -> E4M3 (round to nearest even, saturate to +-448): lo byte = a.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}
// Two E4M3 codes (lo byte = first) -> their values as fp32 (exact).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(uint16_t(two_codes)));
  const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
  return __half22float2(hv);
}
__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  return cvt_e4m3x2(a, b) | (cvt_e4m3x2(c, d) << 16);
}

// |bf16| bit patterns of a packed pair, as an unsigned max-able pair.
__device__ __forceinline__ uint32_t abs2(uint32_t w) { return w & 0x7FFF7FFFu; }
__device__ __forceinline__ uint32_t hmax2(uint32_t w) { return max(w & 0xFFFFu, w >> 16); }

// E8M0 from the bit pattern of a bf16 magnitude (the block maximum):
// exponent field - 8, clamped at 0; Inf or NaN in the block -> 0xFF.
__device__ __forceinline__ uint32_t e8m0_from_bf16abs(uint32_t a) {
  if (a >= 0x7F80u) return 0xFFu;
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

// One 1x32 block of bf16 values held as 16 packed words: its E8M0 scale
// (from the block's largest magnitude), and its 32 E4M3 bytes stored at dst
// (16-byte aligned); a block holding Inf or NaN gets scale 0xFF and 0x7F bytes.
__device__ __forceinline__ uint32_t mx_block_e8m0(const uint32_t* w) {
  uint32_t mx = 0;
#pragma unroll
  for (int e = 0; e < 16; e++) mx = max(mx, hmax2(abs2(w[e])));
  return e8m0_from_bf16abs(mx);
}
__device__ __forceinline__ void mx_block_store(uint8_t* dst, const uint32_t* w, uint32_t sc) {
  uint2 q[4];
  if (sc == 0xFFu) {
#pragma unroll
    for (int v4 = 0; v4 < 4; v4++) q[v4] = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
  } else {
    float inv[8];
    const float f = e8m0_inv_scale(sc);
#pragma unroll
    for (int i = 0; i < 8; i++) inv[i] = f;
#pragma unroll
    for (int v4 = 0; v4 < 4; v4++)
      q[v4] = cvt8(make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]), inv);
  }
  reinterpret_cast<uint4*>(dst)[0] = make_uint4(q[0].x, q[0].y, q[1].x, q[1].y);
  reinterpret_cast<uint4*>(dst)[1] = make_uint4(q[2].x, q[2].y, q[3].x, q[3].y);
}

}  // namespace mxfa
