// qsa_device.cuh -- small device helpers for the sm_103a kernels.
#pragma once

#include <cstdint>
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

}  // namespace qsa
