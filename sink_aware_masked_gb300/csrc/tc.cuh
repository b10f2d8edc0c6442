// Blackwell (sm_100 family, here sm_103a) building blocks written as inline
// PTX: mbarriers with bounded waits, TMA tile loads, Tensor Memory
// allocation, tcgen05.mma (bf16 -> fp32, A from shared or tensor memory),
// tcgen05.commit, and tcgen05.ld / tcgen05.st in the 32x32b shape (thread i
// of a warp <-> TMEM lane 32 * (warp % 4) + i).
//
// Shared-memory operand tiles are 128-byte-swizzled (what a TMA load with
// CU_TENSOR_MAP_SWIZZLE_128B writes): rows of 64 bf16 (128 B), 8-row atoms of
// 1024 B, tile base aligned to 1024 B.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace sa {
namespace tc {

// Status value written to the library's device status word on a timeout
// (equals SINKATTN_ERR_TIMEOUT of the C ABI).
constexpr int kStatusTimeout = 6;
// A wait gives up after this many SM cycles (about one second at 2 GHz).
constexpr long long kTimeoutCycles = 2000000000LL;

// ------------------------------------------------------------------ mbarrier
SA_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
SA_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }
SA_DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
SA_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
SA_DEV void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
SA_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of a phase (try_wait may suspend the thread for a while
// when the phase is still pending; test_wait returns at once).
SA_DEV bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Per-CTA abort word in shared memory plus the global status word.  A wait
// that runs out of time raises both; every later wait in the CTA then fails
// at once, so all warps reach the kernel's exit path promptly.
struct Abort {
  volatile int* flag;  // shared memory
  int* status;         // global device status word
};

// The abort word and the clock are checked on every 16th poll only: the
// shared-memory pipe they use is the one the waiting kernels are short of.
SA_DEV bool mbar_wait(uint32_t bar, uint32_t parity, const Abort& ab, long long limit = kTimeoutCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15) != 0) continue;
    if (*ab.flag) return false;
    if (clock64() - t0 > limit) {
      *ab.flag = 1;
      atomicExch(ab.status, kStatusTimeout);
      return false;
    }
  }
}

// Wait by a whole warp (every lane passes the same barrier and parity).  The
// common case, a phase that has already completed, is a single try_wait and
// a vote with no divergent branch; only a pending phase enters the polling
// loop.
SA_DEV bool mbar_wait_warp(uint32_t bar, uint32_t parity, const Abort& ab) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab));
}

// ------------------------------------------------------------------ TMA
SA_DEV void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
SA_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Brings a tile into L2 ahead of its load (no shared memory, no barrier).
SA_DEV void tma_prefetch_l2_2d(const CUtensorMap* map, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];\n" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}

// Contiguous bulk copy global -> shared on the TMA unit, completing on `bar`
// (both addresses 16-byte aligned, bytes a multiple of 16).
SA_DEV void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}
// Orders this thread's earlier generic-proxy global accesses (and those it
// has acquired) before its later async-proxy (TMA) accesses.
SA_DEV void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;\n" ::: "memory"); }

// 4-byte asynchronous copy global -> shared (Ampere-style cp.async).
SA_DEV void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed;
// the arrival counts toward the barrier's expected count.
SA_DEV void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}
SA_DEV float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];\n" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

// Element-wise atomic add of a shared-memory tile into global memory (fp32).
SA_DEV void tma_reduce_add_2d(const CUtensorMap* map, int c0, int c1, uint32_t src) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];\n" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(src)
      : "memory");
}
// Tile store shared -> global through the tensor map (bulk group; both
// coordinates non-negative, the innermost one 16-byte aligned).
SA_DEV void tma_store_2d(const CUtensorMap* map, int c0, int c1, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];\n" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(src)
               : "memory");
}
SA_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// Wait until the source shared memory of committed bulk groups may be reused.
SA_DEV void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
// Wait until every committed bulk group has completed.
SA_DEV void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

// Named barrier over `n` threads that also returns whether `v` holds for all
// of them: a group that decides together after a bounded wait leaves (or
// stays) together, so none of its threads is left at a later barrier.
SA_DEV bool named_sync_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, %2, %3, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Named barrier over `n` threads that returns whether `v` holds for any of them.
SA_DEV bool named_sync_or(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, %2, %3, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Named barrier over `n` threads (id 1..15; id 0 is __syncthreads).
SA_DEV void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory"); }

// ------------------------------------------------------------------ TMEM
SA_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
SA_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory"); }
SA_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
SA_DEV void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
SA_DEV void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor, 128-byte swizzle, sm_100 format:
// start>>4 in bits 0-13, leading-dimension byte offset>>4 in 16-29,
// stride-dimension byte offset>>4 in 32-45, version 1 in 46-47,
// base offset 0, swizzle mode 2 (128 B) in 61-63.
SA_DEV uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// The same with the swizzle given as the descriptor's layout type (bits
// 61-63): 2 = 128-byte, 4 = 64-byte, 6 = 32-byte swizzle.  For an MN-major
// operand whose swizzle atom spans fewer than 64 bf16 along M or N, the atom
// is 8 rows along K of 64 or 32 bytes (lbo: byte offset between atoms along
// M/N, sbo: between 8-row groups along K).
SA_DEV uint64_t sdesc_swz(uint32_t smem_addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A
// and B (bits 7-9 = 1, 10-12 = 1), operand majorness (bit 15 A, bit 16 B;
// 0 = K-major, 1 = MN-major), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
// Shared-memory matrix descriptor, K-major, no swizzle: 8-row x 16-byte
// core matrices; lbo = byte offset from a core matrix to the next one along
// K, sbo = byte offset between consecutive 8-row groups.
SA_DEV uint64_t sdesc_nosw(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version; layout type 0 (no swizzle) in bits 61-63
  return d;
}

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Advance a shared-memory descriptor's start address by `bytes` (multiple of
// 16; the start field holds address >> 4 and shared addresses stay below
// 256 KB, so the add never carries out of the field).
__host__ __device__ constexpr uint64_t sdesc_add(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

// One elected lane of a converged warp (the lowest active lane).
SA_DEV bool elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n" : "=r"(pred));
  return pred != 0;
}

// ------------------------------------------------------------------ MMA
// D[tmem] (+)= A[smem desc] * B[smem desc]^T ; accumulate when acc != 0.
SA_DEV void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]^T.
SA_DEV void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
SA_DEV void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
               : "memory");
}

// ------------------------------------------------------------------ TMEM <-> registers
#define SA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define SA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
#define SA_F8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])

// 32 consecutive 32-bit columns of this thread's lane.
SA_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : SA_R8(0), SA_R8(8), SA_R8(16), SA_R8(24)
      : "r"(taddr));
}
SA_DEV void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      SA_W8(0), SA_W8(8), SA_W8(16), SA_W8(24)
      : "memory");
}
// 16 consecutive 32-bit columns.
SA_DEV void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : SA_R8(0), SA_R8(8)
      : "r"(taddr));
}
SA_DEV void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr), SA_W8(0)
               : "memory");
}
SA_DEV void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      SA_W8(0), SA_W8(8)
      : "memory");
}
SA_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
SA_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
// Makes the registers filled by tmem_ld32 depend on the preceding wait, so the
// compiler cannot move their first use above tcgen05.wait::ld.
SA_DEV void reg_fence16(uint32_t (&r)[16]) { asm volatile("" : SA_F8(0), SA_F8(8)); }
SA_DEV void reg_fence32(uint32_t (&r)[32]) {
  asm volatile("" : SA_F8(0), SA_F8(8), SA_F8(16), SA_F8(24));
}
#undef SA_R8
#undef SA_W8
#undef SA_F8

// Per-warpgroup register re-allocation (all 4 warps of a warpgroup execute it).
// The sum over warpgroups must stay within the launch's registers
// (threads x registers per thread at launch), or an increase never returns.
template <int N>
SA_DEV void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N));
}
template <int N>
SA_DEV void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N));
}

SA_DEV uint32_t lane_base(int warp) { return static_cast<uint32_t>((warp & 3) * 32) << 16; }

}  // namespace tc
}  // namespace sa
