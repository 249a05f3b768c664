// sv_ptx.cuh -- thin inline-PTX wrappers used by the verify kernels (sm_103a).
//
// Bulk copies (cp.async.bulk) stream each CTA's slice of a logits row from
// HBM into its own shared memory, completing on an mbarrier.
#pragma once

#include <cstdint>

namespace sv {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One arrival that also raises the barrier's expected transaction bytes.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Plain arrival (release at CTA scope: prior shared-memory writes of this
// thread are visible to a thread that then observes the phase completion).
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Named CTA barriers (id 1..15; count: threads taking part, a multiple of
// 32).  sync waits for the barrier; arrive only counts this warp in.  Both
// order the calling threads' earlier shared-memory accesses before the
// threads that then pass the barrier.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void named_bar_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// One wait attempt.  The hint lets the hardware suspend the thread (instead
// of spinning on the issue slot) until the phase completes or ~0.5 ms pass.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(500000u)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Time limit of one bounded wait.  A kernel that has already timed out once
// polls each later barrier only once, so that it drains quickly.
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;

// Wait for the completion of phase `parity` of the barrier.  Gives up after
// kWaitLimitNs and sets `timed_out` (the caller reports a timeout instead of
// hanging).
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, bool& timed_out) {
  if (mbar_try_wait(bar, parity)) return;
  if (timed_out) return;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return;
    if ((i & 3) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
      timed_out = true;
      return;
    }
  }
}

// Non-tensor bulk copy global -> this CTA's shared memory.  dst, src and
// bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 4-byte asynchronous global -> shared copy (cp.async, L1-allocating), and
// its commit / wait groups (hardware waits: they always complete).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- dependent launches
// A kernel launched as a programmatic dependent of the previous kernel on the
// stream may start before that kernel ends; it must wait here before reading
// anything the previous kernel writes.  Without the launch attribute the wait
// returns at once.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the dependent kernel of this one be scheduled as soon as every CTA of
// this grid has executed it (the dependent still waits in grid_dep_wait for
// this grid to finish and its writes to be visible).
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" :::);
}

// ---------------------------------------------------------------- math
// Lane-wise maximum of two bf16 pairs; a NaN in either input gives NaN.
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Hardware base-2 exponential (MUFU); ex2(-inf) = +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max that returns NaN when either input is NaN.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float y;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

}  // namespace sv
