// ra_ring_forward_noalloc: ring attention for callers that cannot allocate.
//
// ra_ring_forward needs a device workspace that the caller allocates.  Some
// callers cannot call cudaMalloc at the point where they run attention: for
// example code on a latency-critical path, where cudaMalloc may synchronise the
// whole device and may fail part-way through a job, or code that runs inside a
// host framework whose allocator owns all device memory and forbids outside
// allocations.  For them this entry point uses a scratch region that the
// library reserves once, in a file-scope device array, and calls nothing that
// allocates (no cudaMalloc, cudaFree, or allocating library routine).
//
// The array is RA_NOALLOC_SCRATCH_BYTES long, and every GPU that loads this
// part of the library keeps it until the process exits.  Problems whose
// workspace would be larger are rejected with RA_ERR_WORKSPACE before anything
// runs.  All calls share the one array and it keeps whatever the previous call
// left there; nothing in it has to start at zero, because every region the
// ring reads is first written by the same call.  Calls whose executions overlap
// on the GPU (different streams, or different host threads on one device)
// race on the array.

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "ra.h"
#include "ra_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[RA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of the scratch array for the current device.  In host code
// the array's name only stands for it; the real address comes from
// cudaGetSymbolAddress, looked up with that device current on the first call
// in each CUDA context (a device reset ends the context, and the next call
// looks the address up again rather than reusing one that no longer exists).
void* scratch_address(cudaError_t* err) {
  struct Entry {
    unsigned long long ctx = 0;
    void* ptr = nullptr;
  };
  static std::mutex mu;
  static Entry cache[kMaxDevices];
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  Entry& e = cache[dev];
  const unsigned long long ctx = ra::current_context_id();
  if (e.ptr == nullptr || e.ctx != ctx) {
    void* ptr = nullptr;
    *err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    e.ptr = ptr;
    e.ctx = ra::current_context_id();
  }
  return e.ptr;
}

}  // namespace

extern "C" ra_status ra_ring_forward_noalloc(const void* q, const void* k, const void* v,
                                             ra_shape shp, int c, int layout, int causal,
                                             int mode, int out_dtype, void* out, float* lse,
                                             ra_stream_t stream) {
  // Empty problems and argument errors are answered by ra_ring_forward
  // itself, before it touches any workspace.
  if (shp.B == 0 || shp.Sq == 0)
    return ra_ring_forward(q, k, v, shp, c, layout, causal, mode, out_dtype, out, lse, nullptr, 0,
                           nullptr, stream);
  const size_t need = ra_ring_forward_workspace_size(shp, c, layout, mode);
  if (need == 0)
    return ra_ring_forward(q, k, v, shp, c, layout, causal, mode, out_dtype, out, lse, nullptr, 0,
                           nullptr, stream);
  if (need > static_cast<size_t>(RA_NOALLOC_SCRATCH_BYTES)) return RA_ERR_WORKSPACE;
  cudaError_t err = cudaSuccess;
  void* scratch = scratch_address(&err);
  if (scratch == nullptr || err != cudaSuccess) return RA_ERR_CUDA;
  return ra_ring_forward(q, k, v, shp, c, layout, causal, mode, out_dtype, out, lse, scratch,
                         static_cast<size_t>(RA_NOALLOC_SCRATCH_BYTES), nullptr, stream);
}
