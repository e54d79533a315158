// Small kernels: the fp32 operand split and the bounded-wait self-test.
#include "spanla_internal.h"
#include "tc_ptx.cuh"

namespace spanla {
namespace {

// x -> (hi, lo) = (bf16(x), bf16(x - bf16(x))), round to nearest even, for
// q, k and v.  Output layout: six [n] bf16 arrays q_hi, q_lo, k_hi, k_lo,
// v_hi, v_lo, back to back.
__global__ void split_f32_kernel(const float4* __restrict__ q, const float4* __restrict__ k,
                                 const float4* __restrict__ v, int64_t n4,
                                 uint2* __restrict__ parts) {
  // The chunk-state kernel may be scheduled now; it waits for this grid's
  // completion before it reads the parts.
  griddep_launch_dependents();
  const float4* src[3] = {q, k, v};
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
#pragma unroll
    for (int t = 0; t < 3; ++t) {
      const float4 x = src[t][i];
      float h0, l0, h1, l1, h2, l2, h3, l3;
      split_bf16(x.x, h0, l0);
      split_bf16(x.y, h1, l1);
      split_bf16(x.z, h2, l2);
      split_bf16(x.w, h3, l3);
      parts[(2 * t) * n4 + i] = make_uint2(pack_bf16x2(h0, h1), pack_bf16x2(h2, h3));
      parts[(2 * t + 1) * n4 + i] = make_uint2(pack_bf16x2(l0, l1), pack_bf16x2(l2, l3));
    }
  }
}

// Waits on an mbarrier that nothing arrives on, with a short limit, then
// records the timeout in the error word and returns.
__global__ void wait_timeout_probe_kernel(unsigned long long limit_ns, unsigned* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(b, 0, limit_ns)) atomicOr(err, kErrTimeoutProbe);
  }
}

}  // namespace

cudaError_t launch_split_f32(const float* q, const float* k, const float* v, int64_t n,
                             void* hi_lo_base, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int64_t n4 = n / 4;   // n = T * H * 64, a multiple of 4
  int64_t blocks = (n4 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  split_f32_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(q), reinterpret_cast<const float4*>(k),
      reinterpret_cast<const float4*>(v), n4, static_cast<uint2*>(hi_lo_base));
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_probe(unsigned limit_us, unsigned* err, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(static_cast<unsigned long long>(limit_us) * 1000ull,
                                                  err);
  return cudaGetLastError();
}

}  // namespace spanla
