// Bulk-copy (TMA) staging primitives for the streaming kernels on sm_100+:
// cp.async.bulk global->shared copies that complete on an mbarrier, and a
// bounded wait on that barrier.
//
// Pipeline shape used by the kernels: a CTA owns S shared-memory stages and
// one mbarrier per stage.  Thread 0 arms a stage's barrier with the bytes it
// expects (arrive.expect_tx) and issues the bulk copies for a tile; all threads
// wait for the barrier's phase, compute from shared memory, and pass a
// __syncthreads() before thread 0 refills the stage with the tile S ahead.  The
// copy engine keeps up to S tiles per CTA in flight without holding registers.
//
// Every wait is bounded (kWaitTimeoutNs of %globaltimer): a wait that runs out
// counts itself in g_pipe_timeouts (one counter per translation unit, read by
// ep_pipeline_timeouts), and the kernel then waits, again bounded, for its
// other copies in flight before it returns, so no copy can land in shared
// memory the CTA no longer owns.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "tuning.h"

namespace ep {
namespace dev {

constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s

static __device__ unsigned int g_pipe_timeouts;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes the initialised barriers visible to the copy engine; follow with __syncthreads().
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

// One test of the phase; the thread may be suspended inside it until the
// phase completes or, with EP_MBAR_SUSPEND_NS > 0, for at most that many ns.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
#if EP_MBAR_SUSPEND_NS > 0
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(uint32_t(EP_MBAR_SUSPEND_NS))
      : "memory");
#else
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
#endif
  return done != 0;
}

// Waits until the barrier's phase with the given parity has completed, for at
// most timeout_ns.  Returns false (and counts a timeout) if it ran out.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > timeout_ns) {
      atomicAdd(&g_pipe_timeouts, 1u);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitTimeoutNs);
}

// Plain arrive (release semantics: this thread's earlier shared-memory reads
// are ordered before the phase completes).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
      : "memory");
}

// A consumer warp hands a stage back to the producer.  The warp's reads of
// the stage go through the generic proxy, the producer's next bulk copy into
// it through the async proxy: a proxy fence orders every lane's reads before
// that copy (without it a copy into a stage whose last reads were still
// queued measured as stale data in the stage's final fragments), then lane 0
// arrives on `empty`.
__device__ __forceinline__ void release_stage(uint64_t* empty_bar) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(empty_bar);
}

// Named barrier over `count` threads (a multiple of 32) with id 1..15; returns
// true on every participating thread iff `pred` held on all of them.
__device__ __forceinline__ bool named_barrier_and(int id, int count, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(uint32_t(pred)), "r"(id), "r"(count)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Evict-first L2 policy for data that is read once.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// global to this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Position in a ring of `n` stages: the stage of the current item and the
// parity of that stage's current use (item i is in stage i % n, use i / n),
// advanced one item at a time without a division.
struct Ring {
  int st = 0;
  uint32_t phase = 0;
  int n;
  __device__ __forceinline__ explicit Ring(int stages) : n(stages) {}
  __device__ __forceinline__ void next() {
    if (++st == n) {
      st = 0;
      phase ^= 1u;
    }
  }
};

// ---------------------------------------------------------------------------
// Dynamic work distribution with cluster launch control (sm_100+).  A kernel
// launched with one CTA per work unit lets each running CTA ask the hardware
// to cancel a CTA of the same grid that has not started yet and take over its
// unit, so SMs that run faster take more units and the grid ends together.
// The 16-byte answer lands in shared memory and completes `bar` with 16
// transaction bytes; after a refusal (no CTA left to cancel) the CTA must not
// ask again.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void clc_try_cancel(void* resp, uint64_t* bar) {
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];"
      ::"r"(smem_addr(resp)), "r"(smem_addr(bar))
      : "memory");
}

// Decodes an answer (16-byte aligned): true, and the x index of the cancelled
// CTA, if a CTA was cancelled.
__device__ __forceinline__ bool clc_query(const void* resp, uint32_t* ctaid_x) {
  uint32_t ok, x;
  asm volatile(
      "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
      "ld.shared.b128 r, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t"
      "mov.u32 %1, 0;\n\t"
      "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
      : "=r"(ok), "=r"(x)
      : "r"(smem_addr(resp))
      : "memory");
  *ctaid_x = x;
  return ok != 0;
}

// Orders this thread's earlier shared-memory accesses before later async-proxy
// (bulk copy, launch control) writes to the same addresses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One thread's stream of work units: this CTA's own unit, then those of the
// CTAs it cancels, with one request kept in flight.  `resp` (16-byte aligned)
// and `bar` (initialised with count 1) are the CTA's.
struct ClcStream {
  void* resp;
  uint64_t* bar;
  uint32_t phase = 0;
  bool pending = false;  // a request is in flight
  __device__ __forceinline__ ClcStream(void* r, uint64_t* b) : resp(r), bar(b) {}
  __device__ __forceinline__ void request() {
    mbar_arrive_expect_tx(bar, 16);
    clc_try_cancel(resp, bar);
    pending = true;
  }
  // The next unit, or -1 when no CTA is left to cancel (or the answer did not
  // come within the bounded wait, which is counted as a timeout).
  __device__ __forceinline__ int64_t next() {
    if (!pending) return -1;
    if (!mbar_wait(bar, phase)) return -1;  // still pending: drain() waits again
    pending = false;
    phase ^= 1u;
    uint32_t x;
    if (!clc_query(resp, &x)) return -1;
    fence_proxy_async_smem();  // the answer is read before the next request overwrites it
    request();
    return int64_t(x);
  }
  // Before the CTA exits: wait (bounded) for a request still in flight.
  __device__ __forceinline__ void drain() {
    if (pending && mbar_wait(bar, phase)) pending = false;
  }
};

// 16-byte shared-memory load.
__device__ __forceinline__ uint4 lds16(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

}  // namespace dev

// Host side: read (and optionally clear) this translation unit's timeout
// counter on the current device.  Synchronous.
static inline cudaError_t read_pipe_timeouts(unsigned int* count, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(count, dev::g_pipe_timeouts, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(dev::g_pipe_timeouts, &zero, sizeof(unsigned int));
}

}  // namespace ep
