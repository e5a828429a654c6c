// qsa_device.cuh -- small device helpers for the sm_103a kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

namespace qsa {

// Packed binary32 fused multiply-add (two IEEE fma.rn lanes in one
// instruction on sm_100-class GPUs): d = a*b + c per component.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 h2f2(uint32_t bits) {
  __half2 h = *reinterpret_cast<__half2*>(&bits);
  return __half22float2(h);
}

// Read-only streaming 16-byte load (no L1 allocation; the line is used once).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before its predecessor finishes; pdl_wait() blocks
// until the predecessor grid has completed and its writes are visible (a
// no-op without the launch attribute).  pdl_trigger() lets the successor be
// scheduled once every CTA of this grid has issued it or exited.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void report(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

// floor division by a positive power-of-two-free constant for int64
__device__ __forceinline__ int64_t floor_div(int64_t a, int64_t b) {
  int64_t q = a / b;
  return (a % b != 0 && a < 0) ? q - 1 : q;
}

// --- mbarriers, TMA and bulk copies (sm_90+ PTX) ---------------------------
//
// Shared-memory operands are 32-bit shared-window addresses.  Every wait on
// a copy or a phase is bounded by the caller's limit, so a lost completion
// can never hang the GPU.

#ifdef QSA_WAIT_TEST
// Test build only (libqsa_waittest.so): waits on a stage give up after 2 ms,
// so a test that withholds one stage's copy sees the timeout path quickly.
constexpr uint64_t kWaitLimitNs = 2000000ull;
#else
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s: any longer wait is a fault
#endif
// Draining copies already in flight after a timeout always gets the full
// second: a copy that was issued lands well within it.
constexpr uint64_t kDrainLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
// arrive and add `bytes` to the phase's expected transaction count
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
               : "memory");
}
// Has the phase of this parity completed?  (A thread whose phase is not
// complete may be held in the instruction for a short, hardware-chosen time.)
__device__ __forceinline__ bool mbar_try_wait(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}
// As mbar_try_wait, suspending the thread up to about hint_ns while the
// phase is incomplete, so waiting warps leave issue slots to working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t a, uint32_t parity,
                                                    uint32_t hint_ns = 20000u) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(a), "r"(parity), "r"(hint_ns) : "memory");
  return ok != 0;
}
// Non-blocking test of a phase (cheaper than try_wait when it has completed).
__device__ __forceinline__ bool mbar_test_wait(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(a), "r"(parity) : "memory");
  return ok != 0;
}
// Wait for the phase of the given parity; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}
// As mbar_wait, with suspended waits (for warps that wait long).
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t a, uint32_t parity) {
  if (mbar_test_wait(a, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait_sleep(a, parity))
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// Tiled TMA loads into shared memory, completing on mbarrier `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x),
      "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x),
      "r"(y), "r"(z), "r"(bar)
      : "memory");
}
// Untiled bulk copy (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

}  // namespace qsa
