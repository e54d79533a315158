// Fixed device scratch for span_la_pass_noalloc.
//
// Some callers cannot allocate device memory while they run a pass: a process
// that hands all of the GPU's memory to its own pool up front, or code that
// runs where an allocation could block or fail at the wrong moment.  For them
// the library keeps one workspace for the whole process in a file-scope device
// array of fixed size.  Every GPU that loads this module holds it until the
// process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "spanla_internal.h"

namespace spanla {
namespace {

// Largest workspace a no-allocation pass may use: descriptors (64 bytes per
// output tile) plus the fp32 64x64 workspace states (16 KiB each).  A piece
// is the part of one view-head (or long-branch-head) inside one CTA's run of
// the output kernel.  The one-launch structure keeps a state only for a piece
// whose state another CTA needs (at most one per boundary between runs), so
// there the descriptors set the limit (about 200,000 tiles); the three-launch
// structure keeps one per piece, at most about (views + SMs) x heads of them
// (a 7,400-token 16-head pass needs about 170, the array about a thousand).
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
// Error word of the no-allocation path's kernels (bounded waits that ran out).
static __device__ unsigned g_noalloc_err;

struct Slot {
  bool ready = false;
  uint8_t* scratch = nullptr;
  unsigned* err = nullptr;
};

std::mutex g_mu;
Slot g_slots[64];

}  // namespace

// Device addresses of the scratch array and error word on the current device.
// The first call on a device looks them up with cudaGetSymbolAddress (with
// that device current) and caches them; later calls only read the cache, so
// the addresses stay valid only while the device's primary context lives (a
// cudaDeviceReset invalidates them).
cudaError_t noalloc_scratch(uint8_t** scratch, unsigned** err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  Slot& s = g_slots[dev];
  if (!s.ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    void* q = nullptr;
    e = cudaGetSymbolAddress(&q, g_noalloc_err);
    if (e != cudaSuccess) return e;
    s.scratch = static_cast<uint8_t*>(p);
    s.err = static_cast<unsigned*>(q);
    s.ready = true;
  }
  *scratch = s.scratch;
  *err = s.err;
  return cudaSuccess;
}

cudaError_t noalloc_error_word(unsigned** err) {
  *err = nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaSuccess;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_slots[dev].ready) *err = g_slots[dev].err;
  return cudaSuccess;
}

}  // namespace spanla
