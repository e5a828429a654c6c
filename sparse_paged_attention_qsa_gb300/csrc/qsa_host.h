// qsa_host.h -- host-side helpers shared by the C ABI entry points.
#pragma once
#include <cuda_runtime.h>

namespace qsa {

// Bind the calling host thread to its current device's primary context for
// this library's (statically linked) CUDA runtime.  In a thread whose CUDA
// work so far went through another copy of the runtime (the caller's
// framework creating its streams, say), launches from this library
// otherwise fail with an invalid-argument error.  Every entry point calls
// this after its host-side checks, before its first other CUDA call.
inline void bind_calling_thread() {
  int d = 0;
  if (cudaGetDevice(&d) == cudaSuccess) cudaSetDevice(d);
}

}  // namespace qsa
