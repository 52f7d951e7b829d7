// Thin inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM alloc, MMA, commit, ld/st) and a bounded mbarrier wait.
//
// Every wait in this library is bounded: after kWaitTimeoutNs of wall time
// (%globaltimer) it raises a CTA-wide abort flag and records an error code in
// the device error word, so a broken pipeline returns instead of hanging.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace attn {

constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s

// Device error codes (written to the per-library device error word).
enum : int {
  kErrNone = 0,
  kErrTimeoutProducer = 0x101,
  kErrTimeoutMma = 0x102,
  kErrTimeoutSoftmax = 0x103,
  kErrTimeoutEpilogue = 0x104,
  kErrTimeoutDiag = 0x105,      // the deliberate wait of ATTN_FWD_DIAG_WAIT_EXPIRES
  kErrTimeoutSelftest = 0x1FF,  // the deliberate wait of attn_selftest_wait_timeout
  kErrDecodeBadBlock = 0x201,
  kErrPagedBadBlock = 0x202,   // paged prefill: block id outside [0, num_blocks)
  kErrPagedBadLength = 0x203,  // paged prefill: kv_lens[b] < 0 or > 16 * max_blocks
  kErrAppendTable = 0x301,     // kv_append: length < 0 or the table is full
  kErrAppendBlock = 0x302,     // kv_append: a table entry is not a block id
  kErrAppendNoFree = 0x303,    // kv_append: not enough free blocks
};

// Where a kernel reports errors.  word[0] holds the first error code any launch
// recorded (kept until attn_device_status reads and clears it); word[1] holds
// the id of the last launch in which a bounded wait expired.  Every launch
// gets a fresh id from the host (never 0), so the skip below stays inside the
// launch that timed out: later launches, and launches running at the same
// time on other streams, do their full work.
struct ErrSink {
  int* word;
  unsigned launch;
  __device__ __forceinline__ void record(int code) const { atomicCAS(word, 0, code); }
  __device__ __forceinline__ void record_timeout(int code) const {
    atomicCAS(word, 0, code);
    atomicExch(reinterpret_cast<unsigned*>(word) + 1, launch);
  }
  // True if a wait of this same launch has already timed out: its later CTAs
  // then skip their work, so one systematic failure costs one timeout, not
  // one per CTA.
  __device__ __forceinline__ bool this_launch_timed_out() const {
    return reinterpret_cast<const volatile unsigned*>(word)[1] == launch;
  }
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase of `bar` with parity `parity` has completed.
// Returns false (without completing) if `abort_flag` is raised by another
// thread, or after limit_ns, in which case it raises the flag itself and
// records `code` (and this launch) in err.
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity,
                                                volatile int* abort_flag, const ErrSink& err,
                                                int code, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        err.record_timeout(code);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          const ErrSink& err, int code) {
  return mbar_wait_limit(bar, parity, abort_flag, err, code, kWaitTimeoutNs);
}

// Drain wait used on the abort path: ignores the abort flag, gives up at the
// absolute %globaltimer deadline shared by all drains of one thread.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t deadline) {
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() > deadline) return false;
  }
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
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

// The tcgen05.mma / tcgen05.commit wrappers below are executed by a whole,
// converged warp; elect.sync picks the one lane that issues.  Issuing from a
// warp-uniform context keeps the descriptors in uniform registers: measured on
// B300, a lane-0-only divergent issue sustained about half the MMA rate.

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc], A held in tensor memory.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Four MMAs of one accumulation chain behind a single elect.sync, from a
// converged warp: D (+)= A_k * B_k for k = 0..3, where operand k sits k * AS
// (A) and k * BS (B) address units past a / b; the first MMA accumulates iff
// acc0 != 0, the other three always.  One elect and one pair of predicate
// setups per four MMAs instead of per MMA: measured on B300 with two
// high-ILP warps sharing the issuing warp's scheduler, issuing eight MMAs
// took 218 cycles this way and 308 with per-MMA elect.
template <int AS, int BS>
__device__ __forceinline__ void mma4_bf16_ss(uint32_t d_tmem, uint64_t a, uint64_t b,
                                             uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, t, e;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      "setp.ne.b32 p, %3, 0;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "add.s64 a1, %1, %5;\n\tadd.s64 a2, %1, %6;\n\tadd.s64 a3, %1, %7;\n\t"
      "add.s64 b1, %2, %8;\n\tadd.s64 b2, %2, %9;\n\tadd.s64 b3, %2, %10;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %4, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %4, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %4, t;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(acc0), "r"(idesc), "n"(AS), "n"(2 * AS), "n"(3 * AS), "n"(BS),
      "n"(2 * BS), "n"(3 * BS)
      : "memory");
}
// The same with A in tensor memory: operand k at TMEM address a + k * AS.
template <int AS, int BS>
__device__ __forceinline__ void mma4_bf16_ts(uint32_t d_tmem, uint32_t a, uint64_t b,
                                             uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, t, e;\n\t.reg .b32 a1, a2, a3;\n\t.reg .b64 b1, b2, b3;\n\t"
      "setp.ne.b32 p, %3, 0;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "add.u32 a1, %1, %5;\n\tadd.u32 a2, %1, %6;\n\tadd.u32 a3, %1, %7;\n\t"
      "add.s64 b1, %2, %8;\n\tadd.s64 b2, %2, %9;\n\tadd.s64 b3, %2, %10;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %4, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %4, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %4, t;\n\t}" ::"r"(d_tmem),
      "r"(a), "l"(b), "r"(acc0), "r"(idesc), "n"(AS), "n"(2 * AS), "n"(3 * AS), "n"(BS),
      "n"(2 * BS), "n"(3 * BS)
      : "memory");
}
// Advance a shared-memory descriptor by `off16` 16-byte units.  The start
// address field is the low 14 bits and every operand here lies below 256 KB,
// so the sum never carries out of the low word: one 32-bit add.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t off16) {
  return (d & 0xFFFFFFFF00000000ull) | uint64_t(uint32_t(d) + off16);
}
// Arrive once on `bar` when every tcgen05 op the issuing lane issued so far is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}
// One elected lane of a converged warp: TMA-load a 3-D box into shared memory
// (signals `bar` on completion).
__device__ __forceinline__ void tma_load_3d_elect(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                                  int c0, int c1, int c2) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// One elected lane of a converged warp: arrive on `bar` expecting `bytes`.
__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
      : "memory");
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, A K-major,
// B K-major (b_mn_major = 0) or MN-major (1); M >> 4 at bit 24, N >> 3 at bit 17.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int b_mn_major) {
  return (1u << 4)        // D format: f32
         | (1u << 7)      // A format: bf16
         | (1u << 10)     // B format: bf16
         | (uint32_t(b_mn_major) << 16) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}
// The same with A from shared memory in MN-major order (bit 15): A's M index
// is the contiguous one, e.g. K^T read from a K tile stored [keys][d].
__host__ __device__ constexpr uint32_t idesc_bf16_f32_amn(int M, int N, int b_mn_major) {
  return idesc_bf16_f32(M, N, b_mn_major) | (1u << 15);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
// lbo / sbo in bytes (leading / stride byte offsets), version bits = 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// 32 lanes x 32 columns of 32-bit from tensor memory (one row per thread).
// Issue only; results are valid after tmem_ld_wait() + reg_fence().
#define ATTN_R32(x) \
  "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), \
  "=r"(x[7]), "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), \
  "=r"(x[14]), "=r"(x[15]), "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), \
  "=r"(x[21]), "=r"(x[22]), "=r"(x[23]), "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), \
  "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31])
#define ATTN_W32(x) \
  "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3]), "r"(x[4]), "r"(x[5]), "r"(x[6]), "r"(x[7]), \
  "r"(x[8]), "r"(x[9]), "r"(x[10]), "r"(x[11]), "r"(x[12]), "r"(x[13]), "r"(x[14]), "r"(x[15]), \
  "r"(x[16]), "r"(x[17]), "r"(x[18]), "r"(x[19]), "r"(x[20]), "r"(x[21]), "r"(x[22]), "r"(x[23]), \
  "r"(x[24]), "r"(x[25]), "r"(x[26]), "r"(x[27]), "r"(x[28]), "r"(x[29]), "r"(x[30]), "r"(x[31])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : ATTN_R32(r)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      ATTN_W32(r)
      : "memory");
}
// 32 lanes x 16 columns of 32-bit into tensor memory (one row per thread).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// tmem_ld32 that also returns, per thread, the maximum of the 32 values it
// loads (tcgen05.ld.red, sm_103a).  Issue only, like tmem_ld32: both are
// valid after tmem_ld_wait() + reg_fence().
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t* r, float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
      : "=f"(*reinterpret_cast<float*>(&r[0])), "=f"(*reinterpret_cast<float*>(&r[1])),
        "=f"(*reinterpret_cast<float*>(&r[2])), "=f"(*reinterpret_cast<float*>(&r[3])),
        "=f"(*reinterpret_cast<float*>(&r[4])), "=f"(*reinterpret_cast<float*>(&r[5])),
        "=f"(*reinterpret_cast<float*>(&r[6])), "=f"(*reinterpret_cast<float*>(&r[7])),
        "=f"(*reinterpret_cast<float*>(&r[8])), "=f"(*reinterpret_cast<float*>(&r[9])),
        "=f"(*reinterpret_cast<float*>(&r[10])), "=f"(*reinterpret_cast<float*>(&r[11])),
        "=f"(*reinterpret_cast<float*>(&r[12])), "=f"(*reinterpret_cast<float*>(&r[13])),
        "=f"(*reinterpret_cast<float*>(&r[14])), "=f"(*reinterpret_cast<float*>(&r[15])),
        "=f"(*reinterpret_cast<float*>(&r[16])), "=f"(*reinterpret_cast<float*>(&r[17])),
        "=f"(*reinterpret_cast<float*>(&r[18])), "=f"(*reinterpret_cast<float*>(&r[19])),
        "=f"(*reinterpret_cast<float*>(&r[20])), "=f"(*reinterpret_cast<float*>(&r[21])),
        "=f"(*reinterpret_cast<float*>(&r[22])), "=f"(*reinterpret_cast<float*>(&r[23])),
        "=f"(*reinterpret_cast<float*>(&r[24])), "=f"(*reinterpret_cast<float*>(&r[25])),
        "=f"(*reinterpret_cast<float*>(&r[26])), "=f"(*reinterpret_cast<float*>(&r[27])),
        "=f"(*reinterpret_cast<float*>(&r[28])), "=f"(*reinterpret_cast<float*>(&r[29])),
        "=f"(*reinterpret_cast<float*>(&r[30])), "=f"(*reinterpret_cast<float*>(&r[31])),
        "=f"(mx)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Ties registers to a point in program order: values loaded by tcgen05.ld are
// only read after the preceding tcgen05.wait::ld.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t* r) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// Per-warpgroup register reallocation (all 4 warps of a warpgroup execute it).
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------ math
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  // cvt packs its first source into the upper half.
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace attn
