// Thin inline-PTX wrappers for the sm_100-family async machinery used by the
// tree-attention kernel: mbarriers, TMA tensor loads, tcgen05 MMA with the
// accumulator in tensor memory (TMEM), TMEM loads/stores and the fences that
// order them.  Written from the PTX ISA's instruction descriptions.
#pragma once

#include <stdint.h>

namespace tsd {
namespace sm100 {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
// One arrival that counts `count` times toward the phase.
__device__ __forceinline__ void mbar_arrive_cnt(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking probe of a phase (no suspend window).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}
// Bounded wait: returns false if the phase did not complete within limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// ---- TMA ------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *tmap, int x, int y, int z,
                                            int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

// L2 prefetch of one tensor box (no shared memory, no completion tracking).
__device__ __forceinline__ void tma_prefetch_4d(const void *tmap, int x, int y, int z, int w) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];\n" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}

// Bulk copy shared -> global (16-byte aligned, size a multiple of 16), and the
// wait for this thread's bulk copies to complete.
// Global -> shared bulk copy completing `bytes` of transaction on `bar`
// (addresses 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t sdst, const void *gsrc, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          sdst),
      "l"(gsrc), "r"(bytes), "r"(bar)
      : "memory");
}
// Bulk prefetch of [gsrc, gsrc + bytes) into L2 (16-byte aligned, bytes a
// multiple of 16); nothing is written to shared memory and nothing waits.
__device__ __forceinline__ void bulk_prefetch_l2(const void *gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(gsrc), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_store(void *gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(gdst),
               "r"(ssrc), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
// L2 policy that evicts the lines it covers after lines of normal priority.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
// bulk_store with an L2 cache policy for the written lines.
__device__ __forceinline__ void bulk_store_hint(void *gdst, uint32_t ssrc, uint32_t bytes,
                                                uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;\n" ::"l"(
                   gdst),
               "r"(ssrc), "r"(bytes), "l"(policy)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
// Drops the 128-byte L2 line at p (128-byte aligned) without writing it back:
// for data that no one will read again.
__device__ __forceinline__ void discard_l2_line(const void *p) {
  asm volatile("discard.global.L2 [%0], 128;\n" ::"l"(p) : "memory");
}
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}
// Wait until this thread's bulk copies have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}

// ---- cp.async (LSU path) with mbarrier completion ------------------------------
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
// The mbarrier receives one arrival when all of this thread's earlier cp.async
// copies have landed (the arrival is counted in the barrier's init count).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;\n" ::: "memory");
}

// ---- proxy / tcgen05 fences --------------------------------------------------
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// ---- TMEM allocation (one full warp) ----------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// ---- UMMA descriptors ---------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (16-byte units), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}
// The descriptor of the matrix `off_bytes` (a multiple of 16) past the one
// `d` describes.  The start-address field holds address / 16 in 14 bits and
// every shared-memory address of a block is below 256 KB, so the sum never
// carries out of the field.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t off_bytes) {
  return d + (uint64_t)(off_bytes >> 4);
}
// Instruction descriptor for kind::f16 with bf16 A/B and an fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major,
                                                      bool b_mn_major) {
  return (1u << 4)                            // D format: f32
         | (1u << 7)                          // A format: bf16
         | (1u << 10)                         // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)     // A major
         | ((b_mn_major ? 1u : 0u) << 16)     // B major
         | ((uint32_t)(N >> 3) << 17)         // N / 8
         | ((uint32_t)(M >> 4) << 24);        // M / 16
}

// ---- tcgen05 MMA ----------------------------------------------------------------
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same, with A (M x K, K-major) read from tensor memory: lane m holds row m,
// each 32-bit column two consecutive K elements (lower index in the low half);
// one K=16 step spans 8 columns.
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Eight MMAs from one asm block (a K = 128 chain of K = 16 steps): D in
// tensor memory, A and B from shared-memory descriptors a[i], b[i].  The first
// step accumulates into D only when acc0 is nonzero, the others always.  One
// block of instructions with its operands in registers keeps the issuing
// thread's instruction count per MMA near one, which matters when the warps
// sharing its SM sub-partition are busy.
__device__ __forceinline__ void umma8_ss(uint32_t d, const uint64_t (&a)[8], const uint64_t (&b)[8],
                                         uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %18, 0;\n setp.ne.b32 q, 1, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %17, p;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %17, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %17, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %17, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %17, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %11, %12, %17, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %13, %14, %17, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %15, %16, %17, q;\n}\n" ::"r"(d),
      "l"(a[0]), "l"(b[0]), "l"(a[1]), "l"(b[1]), "l"(a[2]), "l"(b[2]), "l"(a[3]), "l"(b[3]),
      "l"(a[4]), "l"(b[4]), "l"(a[5]), "l"(b[5]), "l"(a[6]), "l"(b[6]), "l"(a[7]), "l"(b[7]),
      "r"(idesc), "r"(acc0)
      : "memory");
}
// The same with A read from tensor memory: step i reads columns a + 8 i.
__device__ __forceinline__ void umma8_ts(uint32_t d, uint32_t a, const uint64_t (&b)[8],
                                         uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %18, 0;\n setp.ne.b32 q, 1, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %17, p;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %4, %17, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %17, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %17, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %17, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%11], %12, %17, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%13], %14, %17, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%15], %16, %17, q;\n}\n" ::"r"(d),
      "r"(a), "l"(b[0]), "r"(a + 8), "l"(b[1]), "r"(a + 16), "l"(b[2]), "r"(a + 24), "l"(b[3]),
      "r"(a + 32), "l"(b[4]), "r"(a + 40), "l"(b[5]), "r"(a + 48), "l"(b[6]), "r"(a + 56), "l"(b[7]),
      "r"(idesc), "r"(acc0)
      : "memory");
}
// Four steps of the same, A from tensor memory (a K = 64 chain).
__device__ __forceinline__ void umma4_ts(uint32_t d, uint32_t a, const uint64_t (&b)[4],
                                         uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %10, 0;\n setp.ne.b32 q, 1, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %9, p;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %4, %9, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %9, q;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %9, q;\n}\n" ::"r"(d),
      "r"(a), "l"(b[0]), "r"(a + 8), "l"(b[1]), "r"(a + 16), "l"(b[2]), "r"(a + 24), "l"(b[3]),
      "r"(idesc), "r"(acc0)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
      : "memory");
}

// ---- TMEM <-> registers: 32 lanes x 32 consecutive 32-bit columns -------------
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// ---- packed fp32 pairs (two lanes of one 64-bit register pair) ----------------
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long r) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
  return make_float2(a, b);
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// acc_lo += the low bf16 of w and acc_hi += the high one: each is widened to
// fp32 exactly and added with round-to-nearest (PTX mixed-precision add), so
// no shift or mask is needed to unpack the pair.
__device__ __forceinline__ void add_bf16x2(float &acc_lo, float &acc_hi, uint32_t w) {
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n add.rn.f32.bf16 %0, lo, %0;\n"
      " add.rn.f32.bf16 %1, hi, %1;\n}\n"
      : "+f"(acc_lo), "+f"(acc_hi)
      : "r"(w));
}
// max of three floats in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// 2^x with the hardware approximation (PTX ex2.approx.ftz.f32); ex2(-inf) = 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// ---- thread-block clusters ---------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(r));
  return r;
}
// Cluster-wide barrier halves: every thread of every CTA of the cluster
// arrives (release: its earlier shared-memory writes become visible to the
// cluster) and then waits (acquire).  Warp-converged calls only.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// 16-byte load from the shared memory of CTA `rank` of this cluster, at the
// offset that `saddr` has in this CTA's own shared window.
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(saddr), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(r)
               : "memory");
  return v;
}

// 16-byte store into the shared memory of CTA `rank` of this cluster, at the
// offset that `saddr` has in this CTA's own shared window.
__device__ __forceinline__ void st_dsmem_f4(uint32_t saddr, uint32_t rank, float4 v) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(saddr), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(r), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` inside a tile whose rows
// are 128 bytes wide, laid out in the 128-byte swizzle pattern (8-row atoms of
// 1024 bytes, chunk index XOR row-within-atom).  This is the pattern a TMA
// load with 128-byte swizzle writes, and the one the UMMA descriptors above
// describe.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

}  // namespace sm100
}  // namespace tsd
