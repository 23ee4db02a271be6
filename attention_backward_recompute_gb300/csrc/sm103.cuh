// sm_103a building blocks written as inline PTX: mbarriers with bounded waits,
// TMA tile loads, tcgen05 tensor-memory allocation, MMA issue, commit, and
// tensor-memory loads/stores.  Every kernel of the library includes this file.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#ifndef ATTN_WAIT_TIMEOUT_NS
#define ATTN_WAIT_TIMEOUT_NS 1000000000ull   // one second per wait, then give up
#endif

namespace sm103 {

// ----------------------------------------------------------------------------
// error reporting shared by all kernels
// ----------------------------------------------------------------------------
// Device error word codes (OR-ed into the word the host reads back).
enum : uint32_t {
  DEV_ERR_TIMEOUT = 1u,      // a bounded wait gave up
  DEV_ERR_LAYOUT = 8u,       // dynamic shared memory not at the alignment the kernel's layout needs
};

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Arrive once and add `bytes` to the transaction count the phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared abort state of one CTA: a flag in shared memory that any role sets
// when one of its waits times out, so that the other roles stop waiting too,
// plus the global error word the host reads.
struct Abort {
  volatile int* flag;      // shared memory
  uint32_t* err;           // global memory (may be null)
};

__device__ __forceinline__ void raise_error(const Abort& a, uint32_t code) {
  *a.flag = 1;
  if (a.err) atomicOr(a.err, code);
}

// Wait for phase `parity` of `bar` to complete.  Gives up (returns false) when
// the CTA is aborting or after ATTN_WAIT_TIMEOUT_NS, in which case it raises
// DEV_ERR_TIMEOUT.  Never spins forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Abort& a) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_test(bar, parity)) return true;
    if (*a.flag) return false;
    if ((++n & 63u) == 0u && global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) {
      raise_error(a, DEV_ERR_TIMEOUT);
      return false;
    }
  }
}

// Warp-collective wait: every lane waits, and the result is the AND over the
// warp, so a timeout seen by one lane makes the whole warp leave together
// (the tcgen05 loads that follow are warp-collective).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, const Abort& a) {
  const bool ok = mbar_wait(bar, parity, a);
  return __all_sync(0xffffffffu, ok);
}

// Non-blocking test (mbarrier.test_wait never suspends the thread, unlike
// try_wait, which may park it until the phase completes or a time limit).
__device__ __forceinline__ bool mbar_test_now(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking warp-collective test: true when every lane sees the phase
// complete (completion is monotonic, so a false is retried by the caller).
// Used by a warp that polls several barriers, so that one incomplete phase
// does not hold it while another is ready.
__device__ __forceinline__ bool mbar_test_warp(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_test_now(bar, parity));
}

// Bounded polling loop state for a warp that waits on several barriers at
// once: check() returns false (warp-uniformly) once the CTA is aborting or
// ATTN_WAIT_TIMEOUT_NS has passed since the loop began (raising
// DEV_ERR_TIMEOUT in the second case).
struct PollBudget {
  uint64_t t0;
  uint32_t n;
  __device__ __forceinline__ PollBudget() : t0(global_timer_ns()), n(0) {}
  __device__ __forceinline__ bool check(const Abort& a) {
    if (__any_sync(0xffffffffu, *a.flag != 0)) return false;
    if ((++n & 63u) == 0u) {
      if (__any_sync(0xffffffffu, global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS)) {
        raise_error(a, DEV_ERR_TIMEOUT);
        return false;
      }
    }
    return true;
  }
};

// ----------------------------------------------------------------------------
// TMA (tiled bulk tensor copies, global -> shared)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
      "[%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Prefetch a tile into L2 (no shared memory, no barrier): issued a few
// tiles ahead of the tile's real load, so that the load finds its data in L2.
// The same coordinate rules as tma_load_4d apply; out-of-range parts are
// simply not fetched.
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// Generic-proxy writes to shared memory (st.shared) become visible to the
// async proxy (tensor cores, TMA) only after this fence.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------------------
// tcgen05: tensor memory and MMA
// ----------------------------------------------------------------------------
// Allocate `ncols` (power of two, >= 32) tensor-memory columns; the base address
// is written to `*dst_smem`.  Executed by one full warp.
// A kernel that allocates all 512 tensor-memory columns must run one CTA per
// SM: a second resident CTA blocks in tcgen05.alloc until the first frees its
// columns, and the two can wait on each other.  Requesting at least this much
// dynamic shared memory per CTA keeps two of them from sharing an SM (the SM
// has 228 KiB).
constexpr int kSmemOneCtaPerSm = 120 * 1024;

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle.
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-48  descriptor version (1 on sm_100 family)
//   bits 49-51  base offset (0: tiles are 1024-byte aligned)
//   bits 61-63  swizzle mode (2 = 128-byte swizzle)
// K-major operand: rows of 128 bytes (64 bf16 / 32 fp32 of K), 8-row groups
//   SBO = 1024 bytes apart; LBO unused.
// MN-major operand: rows are K, each holding 64 bf16 (32 fp32) of M/N;
//   SBO = 1024 bytes between 8-row K groups, LBO = bytes between successive
//   64-element (128-byte) M/N chunks.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// The same descriptor for an operand without swizzle, in the canonical layout
// of 8-row x 16-byte core matrices (each 128 contiguous bytes).  MN-major:
// a core matrix holds 8 K-rows of 8 bf16 of M/N; LBO = bytes between core
// matrices adjacent along K, SBO = bytes between core matrices adjacent
// along M/N (the reverse of the swizzled MN-major form).
__device__ __forceinline__ uint64_t sdesc_none(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor for kind::f16 (bf16 x bf16 -> f32).
//   bits 4-5 D format (1 = f32); 7-9 A format; 10-12 B format (1 = bf16);
//   15 A MN-major; 16 B MN-major;
//   17-22 N >> 3; 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]; one thread issues.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: A (M x K, bf16 pairs packed two per 32-bit
// column, lower k in the low half; lane = row) is read from tensor memory.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Descriptor of the operand `bytes` further on: only the start-address field
// (address >> 4, 14 bits) changes, and shared-memory addresses stay below
// 256 KB, so the add cannot carry into the other fields.  Lets an issuing
// thread build each descriptor once and step through k-slices with one add.
__device__ __forceinline__ uint64_t sdesc_add(uint64_t desc, uint32_t bytes) {
  return desc + static_cast<uint64_t>(bytes >> 4);
}

// MMA forms with the accumulate flag fixed at compile time (ACC = false:
// D = A*B, the first k-slice; true: D += A*B).  Fewer instructions per MMA
// for the issuing thread, which shares its scheduler with busy warps.
template <bool ACC>
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
  if (ACC)
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 1;" ::"r"(d_tmem), "l"(adesc), "l"(bdesc),
                 "r"(idesc)
                 : "memory");
  else
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 0;" ::"r"(d_tmem), "l"(adesc), "l"(bdesc),
                 "r"(idesc)
                 : "memory");
}
template <bool ACC>
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc) {
  if (ACC)
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 1;" ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc),
                 "r"(idesc)
                 : "memory");
  else
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 0;" ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc),
                 "r"(idesc)
                 : "memory");
}

// Warp-level issue: the whole (converged) warp runs the issuing code and one
// elected lane issues.  With warp-uniform operands the compiler keeps
// descriptors and addresses in uniform registers, so the issuing warp spends
// few instructions per MMA even when the other warps on its scheduler are busy.
template <bool ACC>
__device__ __forceinline__ void mma_ss_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
  if (ACC)
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 1;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 0;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc)
        : "memory");
}
template <bool ACC>
__device__ __forceinline__ void mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc) {
  if (ACC)
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 1;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 0;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc)
        : "memory");
}
// Commit from a converged warp (one elected lane).
__device__ __forceinline__ void mma_commit_w(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_addr(bar))
      : "memory");
}

// Arrive once on `bar` when every MMA issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// Tensor-memory loads: warp w of a warpgroup reads lanes 32*(w%4)..+31; thread
// i gets lane (base lane + i), columns col..col+N-1 (32-bit each).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%"
      "19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
// 32-byte global store (the address must be 32-byte aligned): one full
// sector per thread, half the row requests of two 16-byte stores when the
// threads of a warp write different rows.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]),
               "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// 32 fp32 values of one output row (times f) as bf16, round to nearest even,
// to o[0, valid): 32-byte stores when the whole chunk is in range and o is
// 32-byte aligned, 16-byte stores of 8 values otherwise (o 16-byte aligned).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi);
__device__ __forceinline__ void store_row32_bf16(void* o, const uint32_t (&r)[32], float f, int valid) {
  if (valid >= 32 && (reinterpret_cast<uintptr_t>(o) & 31u) == 0) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        v[e] = pack_bf16x2(__uint_as_float(r[16 * j + 2 * e]) * f, __uint_as_float(r[16 * j + 2 * e + 1]) * f);
      st_global_v8(static_cast<uint8_t*>(o) + 32 * j, v);
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (8 * j < valid) {
      uint4 v;
      v.x = pack_bf16x2(__uint_as_float(r[8 * j]) * f, __uint_as_float(r[8 * j + 1]) * f);
      v.y = pack_bf16x2(__uint_as_float(r[8 * j + 2]) * f, __uint_as_float(r[8 * j + 3]) * f);
      v.z = pack_bf16x2(__uint_as_float(r[8 * j + 4]) * f, __uint_as_float(r[8 * j + 5]) * f);
      v.w = pack_bf16x2(__uint_as_float(r[8 * j + 6]) * f, __uint_as_float(r[8 * j + 7]) * f);
      *reinterpret_cast<uint4*>(static_cast<uint8_t*>(o) + 16 * j) = v;
    }
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ----------------------------------------------------------------------------
// 128-byte-swizzled tile addressing (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B and the MMA reads through sdesc_sw128): a tile is
// rows of 128 bytes; the 16-byte chunk j of row r sits at chunk j ^ (r % 8).
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk16) {
  return row * 128u + (((chunk16 ^ (row & 7u)) & 7u) << 4);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ----------------------------------------------------------------------------
// Packed fp32 pairs: two f32 values in one 64-bit register pair, operated on
// by one instruction; each half is rounded exactly as the scalar operation.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint64_t f2_pack_u(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// bf16 pair (low half = first element) widened to an f32 pair
__device__ __forceinline__ uint64_t f2_from_bf16x2(uint32_t w) { return f2_pack_u(w << 16, w & 0xffff0000u); }
// three-input maximum (a NaN input is ignored, as by fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace sm103
