// Tensor-core rate of the span-output kernel's MMA shapes, on their own.
//
// One elected thread per CTA issues `iters` groups of tcgen05.mma (kind::f16,
// bf16 in, fp32 in tensor memory) back to back from shared-memory operands
// laid out as the kernel lays them out (128-byte swizzle), commits once and
// waits (bounded) for completion.  No loads, no epilogue: the time per group
// is what the tensor pipe needs for that instruction mix.  One CTA per SM.
//
// Modes (per group):
//   qk    4 x M128 N128 K16, A and B K-major           (P = Q K^T of a tile)
//   kv    8 x M128 N64  K16, A and B MN-major          (dS = [K|K]^T V)
//   pv    8 x M128 N64  K16, A from tensor memory      (O = P V)
//   qs    4 x M128 N64  K16, B MN-major                (O += Q S, S in bf16)
//   tile  the 24 of one output tile: qk + kv + pv + qs
//
// Usage: tc_rate <mode> [grid (0: one per SM)] [iters]; prints one line:
//   mode grid iters ns_per_group mhz tflops_per_sm tflops_total err
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>
#include <algorithm>
#include <cuda_runtime.h>
#include "tc_ptx.cuh"

using namespace spanla;

namespace {

constexpr int kSmemBytes = 120 * 1024;   // more than half an SM: one CTA per SM
constexpr uint32_t kOffQ = 0, kOffK = 16384, kOffV = 32768, kOffS = 49152, kOffBar = 65536;

__device__ __forceinline__ uint64_t d_kmajor(uint32_t a, int kk) { return smem_desc_sw128(a + kk * 32, 16, 1024); }
__device__ __forceinline__ uint64_t d_mn(uint32_t a, int kk, uint32_t lbo) {
  return smem_desc_sw128(a + kk * 2048, lbo, 1024);
}

enum Mode { kQK = 0, kKV = 1, kPV = 2, kQS = 3, kTile = 4 };

__global__ void __launch_bounds__(128, 1)
tc_rate_kernel(int mode, int iters, unsigned long long* out, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5;
  // operands: small bf16 values from a hash (their values do not matter)
  for (int i = tid; i < static_cast<int>(kOffBar / 4); i += 128) {
    const uint32_t h = static_cast<uint32_t>(i) * 2654435761u + blockIdx.x * 97u;
    reinterpret_cast<uint32_t*>(smem)[i] =
        pack_bf16x2(((h >> 8) & 0xFFFF) / 65536.0f - 0.5f, ((h >> 3) & 0xFFFF) / 65536.0f - 0.5f);
  }
  fence_proxy_async_smem();
  const uint32_t bar = base + kOffBar;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 16);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(slot), 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *slot;
  if (tid == 0) {
    const uint32_t i_qk = idesc_bf16_f32(128, 128, 0, 0);
    const uint32_t i_kv = idesc_bf16_f32(128, 64, 1, 1);
    const uint32_t i_n64 = idesc_bf16_f32(128, 64, 0, 1);
    const uint32_t q = base + kOffQ, k = base + kOffK, v = base + kOffV, s = base + kOffS;
    const long long c0 = clock64();
    const unsigned long long t0 = global_timer_ns();
    for (int it = 0; it < iters; ++it) {
      const uint32_t b = static_cast<uint32_t>(it & 1);
      const uint32_t colP = b * 128, colO = 256 + b * 64, colD = 384 + b * 64;
      if (mode == kQK || mode == kTile)
        for (int kk = 0; kk < 4; ++kk) mma_bf16(tmem + colP, d_kmajor(q, kk), d_kmajor(k, kk), i_qk, kk > 0);
      if (mode == kKV || mode == kTile)
        for (int kk = 0; kk < 8; ++kk) mma_bf16(tmem + colD, d_mn(k, kk, 0), d_mn(v, kk, 16384), i_kv, kk > 0);
      if (mode == kPV || mode == kTile)
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_tmem_a(tmem + colO, tmem + colP + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8), d_mn(v, kk, 16384),
                          i_n64, kk > 0);
      if (mode == kQS || mode == kTile)
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tmem + colO, d_kmajor(q, kk), d_mn(s, kk, 8192), i_n64, (mode == kTile || kk > 0) ? 1u : 0u);
    }
    mma_commit(bar);
    if (!mbar_wait_bounded(bar, 0, 2000000000ull)) atomicOr(err, 1u);
    const long long c1 = clock64();
    const unsigned long long t1 = global_timer_ns();
    out[blockIdx.x * 2 + 0] = static_cast<unsigned long long>(c1 - c0);
    out[blockIdx.x * 2 + 1] = t1 - t0;
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

int main(int argc, char** argv) {
  const char* names[] = {"qk", "kv", "pv", "qs", "tile"};
  const double flop[] = {4 * 2.0 * 128 * 128 * 16, 8 * 2.0 * 128 * 64 * 16, 8 * 2.0 * 128 * 64 * 16,
                         4 * 2.0 * 128 * 64 * 16, 0};
  int mode = -1;
  for (int m = 0; m < 5; ++m)
    if (argc > 1 && std::strcmp(argv[1], names[m]) == 0) mode = m;
  if (mode < 0) {
    std::fprintf(stderr, "usage: %s qk|kv|pv|qs|tile [grid] [iters]\n", argv[0]);
    return 2;
  }
  int nsm = 0;
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
  int grid = argc > 2 ? std::atoi(argv[2]) : nsm;
  if (grid == 0) grid = nsm;
  const int iters = argc > 3 ? std::atoi(argv[3]) : 256;
  if (grid < 1 || grid > nsm || iters < 1 || iters > (1 << 20)) {
    std::fprintf(stderr, "grid must be in [1, %d], iters in [1, 2^20]\n", nsm);
    return 2;
  }
  cudaFuncSetAttribute(tc_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  unsigned long long* d_out = nullptr;
  unsigned* d_err = nullptr;
  if (cudaMalloc(&d_out, sizeof(unsigned long long) * 2 * grid) != cudaSuccess ||
      cudaMalloc(&d_err, sizeof(unsigned)) != cudaSuccess) {
    std::fprintf(stderr, "cudaMalloc failed\n");
    return 1;
  }
  cudaMemset(d_err, 0, sizeof(unsigned));
  for (int rep = 0; rep < 2; ++rep) tc_rate_kernel<<<grid, 128, kSmemBytes>>>(mode, iters, d_out, d_err);
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    std::fprintf(stderr, "CUDA error: %s\n", cudaGetErrorString(e));
    return 1;
  }
  std::vector<unsigned long long> h(2 * grid);
  unsigned herr = 0;
  cudaMemcpy(h.data(), d_out, sizeof(unsigned long long) * 2 * grid, cudaMemcpyDeviceToHost);
  cudaMemcpy(&herr, d_err, sizeof(unsigned), cudaMemcpyDeviceToHost);
  std::vector<double> ns, mhz;
  for (int c = 0; c < grid; ++c) {
    ns.push_back(static_cast<double>(h[2 * c + 1]) / iters);
    mhz.push_back(static_cast<double>(h[2 * c]) / static_cast<double>(h[2 * c + 1]) * 1e3);
  }
  std::sort(ns.begin(), ns.end());
  std::sort(mhz.begin(), mhz.end());
  const double ns_med = ns[ns.size() / 2];
  const double f = mode == 4 ? flop[0] + flop[1] + flop[2] + flop[3] : flop[mode];
  const double tf_sm = f / ns_med / 1e3;
  std::printf("%s %d %d %.2f %.0f %.3f %.1f %u\n", names[mode], grid, iters, ns_med, mhz[mhz.size() / 2], tf_sm,
              tf_sm * grid, herr);
  return herr == 0 ? 0 : 1;
}
