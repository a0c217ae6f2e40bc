// Inline-PTX building blocks for sm_103a kernels: mbarriers with bounded
// waits, TMA tile loads, tcgen05 MMA / TMEM traffic and the shared-memory
// and instruction descriptors that tcgen05.mma reads.
//
// Every wait in this library is bounded: a wait that outlives its limit sets
// a shared abort flag and the library's device status word, and the caller
// unwinds (drains its own copies and MMAs, frees TMEM) instead of spinning.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "upipe_internal.h"

namespace upipe {

// --------------------------------------------------------------- addresses

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// SM cycle counter, used to bound waits.  It is cheap to read, unlike
// %globaltimer, whose read can hold a polling warp for about a thousand
// cycles and so delay its noticing a completed barrier phase.  Limits are
// given in nanoseconds and compared against cycles at an assumed clock of at
// most 3 GHz, so a wait lasts at least its limit in wall time at any real
// SM clock.
__device__ __forceinline__ uint64_t sm_cycles() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t));
  return t;
}
constexpr uint64_t kCyclesPerNs = 3;

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

// kCluster: acquire at cluster scope, for phases completed by arrivals or
// copies from the other CTA of a pair.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (kCluster) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  }
  return ok != 0;
}

// Non-blocking probe: true iff the phase of parity `parity` has completed.
// (try_wait may suspend the thread for a while; a thread that polls several
// barriers and issues whichever is ready must not block on any one of them.)
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (kCluster) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  }
  return ok != 0;
}

// Per-CTA wait control: the shared abort flag, the device status word and
// the time limit of one wait.
struct WaitCtl {
  volatile int* abort_flag;  // shared memory
  int* status;               // global status word
  uint64_t limit_ns;
};

// Waits for the phase of parity `parity` of barrier `bar`.  Returns false if
// the wait gave up: its own limit ran out (this thread then raises the abort
// flag and records a timeout) or another thread of the CTA aborted first.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  if (mbar_try_wait<kCluster>(bar, parity)) return true;
  const uint64_t t0 = sm_cycles();
  while (true) {
    if (mbar_try_wait<kCluster>(bar, parity)) return true;
    if (*w.abort_flag) return false;
    if (sm_cycles() - t0 > w.limit_ns * kCyclesPerNs) {
      *w.abort_flag = 1;
      atomicOr(w.status, UPIPE_STATUS_TIMEOUT);
      return false;
    }
  }
}

// Bounded wait that spins on the non-blocking probe instead of try_wait, for
// a thread whose next action is latency-critical (an MMA issuer): no
// suspend/wake-up between the phase completing and the thread noticing.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_spin(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  uint64_t t0 = 0;
  for (uint32_t i = 1;; ++i) {
    if (mbar_test<kCluster>(bar, parity)) return true;
    if ((i & 31) != 0) continue;  // the abort flag and the clock every 32 polls
    if (*w.abort_flag) return false;
    const uint64_t now = sm_cycles();
    if (i == 32) {
      t0 = now;
    } else if (now - t0 > w.limit_ns * kCyclesPerNs) {
      *w.abort_flag = 1;
      atomicOr(w.status, UPIPE_STATUS_TIMEOUT);
      return false;
    }
  }
}

// Drain wait used while unwinding: ignores the abort flag, bounded by a fixed
// limit.  Used only on events that complete without help from other threads
// (TMA bytes landing, issued MMAs retiring).
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, int* status) {
  const uint64_t t0 = sm_cycles();
  while (!mbar_try_wait<kCluster>(bar, parity)) {
    if (sm_cycles() - t0 > 1000000000ull * kCyclesPerNs) {
      atomicOr(status, UPIPE_STATUS_DRAIN_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Warp-wide wait: every lane probes the barrier each round and the warp moves
// on once all lanes have seen the phase complete (each lane's own probe is
// its acquire).  Free of divergence on purpose: a lane-0 poll loop followed
// by a broadcast costs about 200 cycles even on a phase that completed long
// ago, against about 15 for one warp-wide probe.  The abort flag and the
// clock are checked every 32 rounds, by warp vote.  Must be called by all 32
// lanes; the result is warp-uniform.
//
// kSuspend probes with try_wait, which suspends the warp in hardware until
// the phase completes (or a system time limit passes) instead of spinning:
// for warps that wait long and often (the backward kernels' compute warps),
// spinning probes took a third of the load/store issue slots and competed
// for issue slots with the MMA-issuing threads on the same sub-partitions.
template <bool kCluster = false, bool kSuspend = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  uint64_t t0 = 0;
  for (uint32_t i = 1;; ++i) {
    const bool done = kSuspend ? mbar_try_wait<kCluster>(bar, parity) : mbar_test<kCluster>(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if (!kSuspend && (i & 31) != 0) continue;
    if (__any_sync(0xffffffffu, *w.abort_flag != 0)) return false;
    const uint64_t now = sm_cycles();
    if (i == (kSuspend ? 1u : 32u)) {
      t0 = now;
    } else if (__any_sync(0xffffffffu, now - t0 > w.limit_ns * kCyclesPerNs)) {
      if ((threadIdx.x & 31) == 0) {
        *w.abort_flag = 1;
        atomicOr(w.status, UPIPE_STATUS_TIMEOUT);
      }
      __syncwarp();
      return false;
    }
  }
}

// No-progress watchdog for a thread that polls several barriers with
// non-blocking probes and issues whatever is ready: `alive` turns false
// (raising the abort flag and the timeout status) once `limit_ns` passes
// without progress, or as soon as another thread of the CTA aborted.  The
// abort flag and the clock are read only every 32 idle polls, so that a poll
// that finds work ready reacts within a few cycles.
struct Watchdog {
  uint64_t t0;
  uint32_t idle;
  __device__ __forceinline__ void reset() { idle = 0; }
  __device__ __forceinline__ bool alive(const WaitCtl& w) {
    if ((++idle & 31) != 0) return true;  // the abort flag and the clock every 32 idle polls
    if (*w.abort_flag) return false;
    const uint64_t now = sm_cycles();
    if (idle == 32) {
      t0 = now;
    } else if (now - t0 > w.limit_ns * kCyclesPerNs) {
      *w.abort_flag = 1;
      atomicOr(w.status, UPIPE_STATUS_TIMEOUT);
      return false;
    }
    return true;
  }
};

// --------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads (tcgen05.mma operands).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ------------------------------------------------------ CTA pairs (cluster of 2)
//
// A pair of CTAs on two SMs runs one M=256 product: the even CTA's thread
// issues tcgen05.mma.cta_group::2, each CTA supplies 128 rows of A and half
// of B's N from its own shared memory at the same offsets, and each CTA's
// TMEM receives its own 128 rows of D.

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of both CTAs; used only where every thread arrives promptly
// (after barrier initialisation, and at exit once every bounded wait has
// returned).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared::cluster address of `addr` (a shared::cta address) in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
// Posts the byte count of copies that will complete on `cluster_bar`.
// Relaxed: it publishes no data of this thread (the copies' completion is
// tracked by the barrier's transaction count); a release here would wait
// for this thread's earlier copies and serialise the ring.
__device__ __forceinline__ void mbar_expect_tx_cluster(uint32_t cluster_bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Tile copies into this CTA's shared memory that complete on a barrier of
// either CTA of the pair (`cluster_bar`, a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t cluster_bar, int c0,
                                                 int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(dst),
      "l"(map), "r"(cluster_bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t cluster_bar, int c0,
                                                 int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, "
      "%5}], [%2];" ::"r"(dst),
      "l"(map), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T.  A is K-major in TMEM: lane r holds row
// r, 32-bit column c holds elements (2c, 2c+1) of that row (low half first),
// so one K=16 step reads 8 columns.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A * B^T over a CTA pair (M = 256); issued by the even CTA.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on the barrier at offset `bar` in every CTA of `mask` when
// every pair product issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, dense.
// a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                          // D format: f32
         | (1u << 7)                        // A format: bf16
         | (1u << 10)                       // B format: bf16
         | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.  For a K-major operand
// `sbo` is the distance between 8-row groups (1024 for dense 128-byte rows)
// and `lbo` is unused; for an MN-major operand `lbo` is the distance between
// 64-element MN groups and `sbo` between 8-row K groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // tcgen05 descriptor version
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// TMEM address of (lane quadrant of this warp, column).
__device__ __forceinline__ uint32_t tmem_lane_addr(uint32_t base, int warp_quadrant, int col) {
  return base + (static_cast<uint32_t>(warp_quadrant * 32) << 16) + static_cast<uint32_t>(col);
}

#define UPIPE_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define UPIPE_P8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])
#define UPIPE_S8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive TMEM columns of this thread's lane -> 32 registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : UPIPE_R8(0), UPIPE_R8(8), UPIPE_R8(16), UPIPE_R8(24)
      : "r"(taddr)
      : "memory");
}

// Waits for this thread's tcgen05.ld; the registers are threaded through so
// that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : UPIPE_P8(0), UPIPE_P8(8), UPIPE_P8(16), UPIPE_P8(24)::"memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : UPIPE_R8(0), UPIPE_R8(8)
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : UPIPE_P8(0), UPIPE_P8(8)::"memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      UPIPE_S8(0), UPIPE_S8(8), UPIPE_S8(16), UPIPE_S8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Copies this thread's 128-element bf16 row of a [128][128] tile that TMA
// wrote with 128-byte swizzle (two 64-column halves of 16 KB) into 64 TMEM
// columns as packed pairs -- the layout tcgen05.mma reads an A operand in.
__device__ __forceinline__ void tile_row_to_tmem(uint32_t tile, int r, uint32_t taddr) {
#pragma unroll
  for (int hq = 0; hq < 2; ++hq) {
    uint32_t q[32];
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      uint32_t a = tile + hq * 16384 + static_cast<uint32_t>(r * 128 + ((ch ^ (r & 7)) << 4));
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(q[4 * ch]), "=r"(q[4 * ch + 1]), "=r"(q[4 * ch + 2]), "=r"(q[4 * ch + 3])
                   : "r"(a));
    }
    tmem_st32(taddr + hq * 32, q);
  }
}

// ------------------------------------------------------------------ misc

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Paired fp32 arithmetic (two lanes of fp32 in one 64-bit register pair),
// which halves the issue slots of the softmax element-wise math.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Stores v[0..7] as bf16 at p.  With lo_off != 0 it also stores the
// rounding residuals v - bf16(v), rounded to bf16, at p + lo_off: the pair
// (high, low) carries about 16 significant bits of each fp32 value.
__device__ __forceinline__ void store8_bf16_split(__nv_bfloat16* p, const float* v, int64_t lo_off) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 hb = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
    h[e] = *reinterpret_cast<const uint32_t*>(&hb);
    const float2 hf = __bfloat1622float2(hb);
    l[e] = pack_bf16x2(v[2 * e] - hf.x, v[2 * e + 1] - hf.y);
  }
  st_global_v4(p, h[0], h[1], h[2], h[3]);
  if (lo_off) st_global_v4(p + lo_off, l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Byte offset of 16-byte chunk `ch` (0..7) of row `r` inside a 128-byte
// swizzled tile of dense 128-byte rows (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B and tcgen05.mma reads with 128-byte swizzle).
__device__ __forceinline__ uint32_t sw128_offset(int r, int ch) {
  return static_cast<uint32_t>(r * 128 + ((ch ^ (r & 7)) << 4));
}

}  // namespace upipe
