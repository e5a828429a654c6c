// qsa_host.h -- host-side helpers shared by the C ABI entry points.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace qsa {

// Driver entry points, resolved once through the runtime (no link-time
// dependency on the driver library).
struct CtxFns {
  CUresult (*get_current)(CUcontext*) = nullptr;
  CUresult (*device_get)(CUdevice*, int) = nullptr;
  CUresult (*primary_retain)(CUcontext*, CUdevice) = nullptr;
  CUresult (*primary_release)(CUdevice) = nullptr;
  CUresult (*primary_state)(CUdevice, unsigned*, int*) = nullptr;
  bool ok = false;
};

inline const CtxFns& ctx_fns() {
  static const CtxFns fns = [] {
    CtxFns f;
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<CUresult (*)(CUcontext*)>(p);
    if (cudaGetDriverEntryPointByVersion("cuDeviceGet", &p, 2000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.device_get = reinterpret_cast<CUresult (*)(CUdevice*, int)>(p);
    if (cudaGetDriverEntryPointByVersion("cuDevicePrimaryCtxRetain", &p, 7000, cudaEnableDefault,
                                         &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.primary_retain = reinterpret_cast<CUresult (*)(CUcontext*, CUdevice)>(p);
    if (cudaGetDriverEntryPointByVersion("cuDevicePrimaryCtxRelease", &p, 11000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.primary_release = reinterpret_cast<CUresult (*)(CUdevice)>(p);
    if (cudaGetDriverEntryPointByVersion("cuDevicePrimaryCtxGetState", &p, 7000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.primary_state = reinterpret_cast<CUresult (*)(CUdevice, unsigned*, int*)>(p);
    f.ok = f.get_current && f.device_get && f.primary_retain && f.primary_release &&
           f.primary_state;
    cudaGetLastError();
    return f;
  }();
  return fns;
}

// Bind the calling host thread to its current device's primary context for
// this library's (statically linked) CUDA runtime.  In a thread whose CUDA
// work so far went through another copy of the runtime (the caller's
// framework creating its streams, say), launches from this library
// otherwise fail with an invalid-argument error.  A context the caller made
// current itself (not the device's primary one) is left current.  Every
// entry point calls this after its host-side checks, before its first other
// CUDA call.
inline void bind_calling_thread() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  const CtxFns& f = ctx_fns();
  if (!f.ok) return;
  CUcontext cur = nullptr;
  if (f.get_current(&cur) != CUDA_SUCCESS) return;
  static thread_local CUcontext bound = nullptr;   // this thread's last bound context
  if (cur != nullptr && cur == bound) return;
  if (cur != nullptr) {
    // is the current context the device's primary one?  (An inactive
    // primary context cannot be current; retaining one only to compare would
    // create it.)
    CUdevice dev = 0;
    unsigned flags = 0;
    int active = 0;
    if (f.device_get(&dev, d) != CUDA_SUCCESS ||
        f.primary_state(dev, &flags, &active) != CUDA_SUCCESS || !active)
      return;
    CUcontext prim = nullptr;
    if (f.primary_retain(&prim, dev) != CUDA_SUCCESS) return;
    const bool primary = prim == cur;
    f.primary_release(dev);
    if (!primary) return;              // the caller's own context
  }
  if (cudaSetDevice(d) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  if (f.get_current(&cur) == CUDA_SUCCESS) bound = cur;
}

}  // namespace qsa
