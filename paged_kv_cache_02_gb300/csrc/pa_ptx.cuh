// pa_ptx.cuh -- inline-PTX helpers for sm_103a: mbarriers, TMA, bounded waits.
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Records the first device-side error (first writer wins) and never traps.
__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-suspending probe of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete. Gives up after limit_ns
// (default about one second), records PA_DEVERR_TIMEOUT and returns false. The
// pipeline waits of the attention kernels take the call's limit (AttnArgs::wait_ns);
// the waits of an abort path (for the CTA's own copies and MMAs in flight) always
// take the default, so that nothing the CTA issued is still running when it exits.
// try_wait may suspend the thread for a hardware-chosen while before it reports a
// phase still open, so a bound shorter than kShortWaitNs polls with the
// non-suspending probe instead, which keeps such a bound exact (it exists to test
// the timeout path).
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint64_t kShortWaitNs = 100000ull;
// the short-bound path, kept out of line: it never runs in a normal call
static __device__ __noinline__ bool mbar_wait_short(uint32_t a, uint32_t parity, int* err,
                                             uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test_wait(a, parity)) {
    if (global_timer_ns() - t0 > limit_ns) {
      record_error(err, PA_DEVERR_TIMEOUT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err,
                                          uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_addr(bar);
  if (limit_ns < kShortWaitNs) return mbar_wait_short(a, parity, err, limit_ns);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(a, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      record_error(err, PA_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// Bound of a kernel's pipeline waits. The kernels are built twice: with kShortWaits
// false the bound is the compile-time default (the build every normal call runs); with
// true it is the call's bound (AttnArgs::wait_ns), selected only by a plan whose wait
// bound differs from the default -- the tests of the timeout path.
template <bool kShortWaits, class Args>
__device__ __forceinline__ uint64_t wait_bound(const Args& a) {
  if constexpr (kShortWaits) return a.wait_ns;
  else return kWaitLimitNs;
}

// mbar_wait executed by every lane of a warp, with one verdict for the whole warp:
// warp-collective instructions that follow (shuffles, ballots, tcgen05.ld / st)
// then never see a warp split by a wait that ran out in some lanes only.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, int* err,
                                               uint64_t limit_ns = kWaitLimitNs) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, err, limit_ns));
}

// 3-D tiled TMA load into shared memory, completing on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

// 5-D tiled TMA load into shared memory, completing on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(smem_addr(bar))
      : "memory");
}

// 3-D tiled TMA store from shared memory (bulk-group completion: the issuing thread
// commits and waits for its own groups).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the thread's bulk stores have read their shared-memory source
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// the thread's bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch: let the next kernel of the stream start its CTAs
// (when it was launched as a programmatic dependent), and wait until the kernel this
// one depends on has completed with its memory visible (a no-op otherwise).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Named barrier over `count` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---- block-table cache of a producer warp.
// An item's block ids (logical blocks first .. first + count - 1 of its row) are
// loaded into registers one item ahead (16 per lane, 512 per item) and stored to
// shared memory when the producer reaches that item, so that issuing a tile only
// reads shared memory. Ids past the cached 512 are read from global memory.
constexpr int kBtCache = 512;
constexpr int kBtPerLane = kBtCache / 32;

struct BtWindow {
  int first;  // first logical block held
  int count;  // number of logical blocks the item needs
};

__device__ __forceinline__ BtWindow bt_window(int kv_begin, int kv_end, int block_size) {
  BtWindow w;
  w.first = kv_begin / block_size;
  w.count = (kv_end - 1) / block_size - w.first + 1;
  return w;
}

// Loads (into registers) the cached part of an item's block ids; -2 marks an index
// past the table row, -3 an unused slot.
__device__ __forceinline__ void bt_prefetch(const int32_t* bt_row, int max_blocks, BtWindow w,
                                            int lane, int (&r)[kBtPerLane]) {
#pragma unroll
  for (int i = 0; i < kBtPerLane; ++i) {
    const int idx = lane + 32 * i;
    const int lb = w.first + idx;
    r[i] = (idx >= w.count) ? -3 : (lb < max_blocks ? __ldg(bt_row + lb) : -2);
  }
}

__device__ __forceinline__ void bt_store(int* cache, const int (&r)[kBtPerLane], int lane) {
#pragma unroll
  for (int i = 0; i < kBtPerLane; ++i) cache[lane + 32 * i] = r[i];
}

// Block id of logical block lb of the item (cache first, global memory beyond it);
// -2 if lb is past the table row.
__device__ __forceinline__ int bt_lookup(const int* cache, BtWindow w, const int32_t* bt_row,
                                         int max_blocks, int lb) {
  const int idx = lb - w.first;
  if (idx < kBtCache) return cache[idx];
  return lb < max_blocks ? __ldg(bt_row + lb) : -2;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- packed pairs of fp32 (one instruction for two lanes of arithmetic, sm_100 family)
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
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
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// max of three floats in one instruction (sm_100 family)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

}  // namespace pa
