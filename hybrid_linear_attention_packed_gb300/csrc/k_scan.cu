// Segmented scan kernel: one exclusive prefix scan of local states across
// every segment of the pass, in a single launch.
//
// "Serving 0.88M TPS from Two RTXs and Mac Minis", section "Kernels": one scan
// covers every view in a pass instead of one scan per view (the second of the
// three launches).  For a run of state slots c0 .. c0+n-1 (the chunks of one
// segment, or the pieces of one segment-head) it replaces slot c by
// sum_{c' < c} dS_{c'}  (the state entering chunk or piece c) and writes the
// run's total (the view's final state) to final_out[final_idx] when
// final_idx >= 0.  An empty view (n = 0) gets the zero state.
//
// fp32 adds on CUDA cores; the kernel is bound by memory traffic.  One CTA of
// 128 threads owns a 512-float eighth of one (segment, head) state and walks
// the run in order, keeping the running sum in registers and loading
// thirty-two slots ahead so the loads stay in flight while the stores drain.
#include "spanla_internal.h"
#include "tc_ptx.cuh"

namespace spanla {
namespace {

constexpr int kThreads = 128;
constexpr int kSlices = kStateFloats / (kThreads * 4);   // 8 CTAs per (segment, head)
constexpr int kAhead = 32;

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

__global__ void __launch_bounds__(kThreads)
segmented_scan_kernel(const ScanDesc* __restrict__ scan, int H, float* __restrict__ ws,
                      float* __restrict__ final_out) {
  // The next kernel may be scheduled now: it waits for this grid's completion
  // before it reads anything written here.
  griddep_launch_dependents();
  griddep_wait();   // chunk states from the previous kernel
  const ScanDesc sd = scan[blockIdx.x];
  // Chunk mode: slot c of head h at (slot0 + c) * H + h.  Span mode: one
  // head per entry, slot c at slot0 + c.
  const bool one_head = sd.head >= 0;
  const int h = one_head ? sd.head : blockIdx.y;
  const int off = (blockIdx.z * kThreads + threadIdx.x) * 4;
  const int64_t stride = one_head ? kStateFloats : static_cast<int64_t>(H) * kStateFloats;
  float* p = ws + (one_head ? static_cast<int64_t>(sd.slot0) : static_cast<int64_t>(sd.slot0) * H + h) *
                      kStateFloats + off;

  float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < sd.nslots; c0 += kAhead) {
    float4 x[kAhead];
#pragma unroll
    for (int j = 0; j < kAhead; ++j)
      if (c0 + j < sd.nslots) x[j] = *reinterpret_cast<const float4*>(p + (c0 + j) * stride);
#pragma unroll
    for (int j = 0; j < kAhead; ++j) {
      if (c0 + j < sd.nslots) {
        *reinterpret_cast<float4*>(p + (c0 + j) * stride) = run;
        run = add4(run, x[j]);
      }
    }
  }
  if (sd.final_idx >= 0) {
    float* f = final_out + (static_cast<int64_t>(sd.final_idx) * H + h) * kStateFloats + off;
    *reinterpret_cast<float4*>(f) = run;
  }
}

}  // namespace

cudaError_t launch_scan(const ScanDesc* scan, int n_scan, int H, bool span_mode, float* ws,
                        float* final_out, cudaStream_t stream, bool pdl) {
  if (n_scan <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_scan, span_mode ? 1 : H, kSlices);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, segmented_scan_kernel, scan, H, ws, final_out);
}

}  // namespace spanla
