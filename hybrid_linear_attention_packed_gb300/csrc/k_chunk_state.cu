// Chunk-state kernel: the local state dS_c = K_c^T V_c of every 64-row chunk.
//
// "Serving 0.88M TPS from Two RTXs and Mac Minis", section "Kernels": linear
// attention runs in 64-token chunks, each needing a few 64x64 matrix products;
// this is the first of the three launches of one scan per pass.
//
// One CTA (128 threads) handles one chunk for two adjacent heads h0, h0+1.
// TMA brings K and V of both heads in as [head][64 rows][64 d] bf16 tiles with
// the 128-byte swizzle.  The contraction runs over tokens, which is the row
// (non-contiguous) dimension of both tiles, so both operands are MN-major:
//   A (M = 128) = [K_h0 | K_h1]^T : the two heads are the two 64-wide M atoms,
//   B (N = 64)  = V_h              : one per head,
// giving D_h = [K_h0^T V_h ; K_h1^T V_h]; rows 64*h .. 64*h+63 of D_h are the
// wanted K_h^T V_h.  Accumulation is fp32 in TMEM.  fp32 inputs arrive as
// bf16 high/low parts and use three products (hi*hi + hi*lo + lo*hi).
// Rows past the chunk's length are zeroed in shared memory before the MMAs,
// so the next segment's rows that the fixed-size box also fetched contribute
// nothing.
#include "spanla_internal.h"
#include "tc_ptx.cuh"

namespace spanla {
namespace {

constexpr int kThreads = 128;
constexpr uint32_t kHeadTileBytes = kChunk * 128;               // 64 rows x 128 B
constexpr uint32_t kOperandBytes = kChunkBoxHeads * kHeadTileBytes;  // 16 KiB
constexpr uint32_t kTmemCols = 128;

template <int SPLIT>
struct ChunkSmem {
  static constexpr uint32_t kK = 0;                              // K parts
  static constexpr uint32_t kV = kK + SPLIT * kOperandBytes;     // V parts
  static constexpr uint32_t kBar = kV + SPLIT * kOperandBytes;   // 2 mbarriers
  static constexpr uint32_t kTmemSlot = kBar + 16;
  static constexpr uint32_t kBytes = kTmemSlot + 16;
  // Requested dynamic shared memory: the layout, 1 KiB of alignment slack,
  // and padding that keeps at most 4 CTAs (4 x 128 TMEM columns) per SM.
  static constexpr uint32_t kRequest = (kBytes + 1024 > 58 * 1024) ? kBytes + 1024 : 58 * 1024;
};

template <int SPLIT>
__global__ void __launch_bounds__(kThreads)
chunk_state_kernel(const __grid_constant__ CUtensorMap tm_k0, const __grid_constant__ CUtensorMap tm_k1,
                   const __grid_constant__ CUtensorMap tm_v0, const __grid_constant__ CUtensorMap tm_v1,
                   const ChunkDesc* __restrict__ chunks, int H, float* __restrict__ ws,
                   unsigned* __restrict__ err) {
  using L = ChunkSmem<SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int chunk = blockIdx.x;
  const int h0 = blockIdx.y * kChunkBoxHeads;
  const ChunkDesc cd = chunks[chunk];

  const uint32_t bar_tma = base + L::kBar;
  const uint32_t bar_mma = base + L::kBar + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();                 // the bf16 parts from the split kernel
  griddep_launch_dependents();    // the scan waits for this grid itself

  if (tid == 0) {
    mbar_arrive_expect_tx(bar_tma, 2 * SPLIT * kOperandBytes);
    tma_load_3d(base + L::kK, &tm_k0, bar_tma, 0, cd.row0, h0);
    tma_load_3d(base + L::kV, &tm_v0, bar_tma, 0, cd.row0, h0);
    if (SPLIT == 2) {
      tma_load_3d(base + L::kK + kOperandBytes, &tm_k1, bar_tma, 0, cd.row0, h0);
      tma_load_3d(base + L::kV + kOperandBytes, &tm_v1, bar_tma, 0, cd.row0, h0);
    }
  }

  bool ok = mbar_wait_bounded(bar_tma, 0, kWaitLimitNs);
  if (!ok) {
    atomicOr(err, kErrTimeoutTma);
    mbar_wait_bounded(bar_tma, 0, kWaitLimitNs);  // let copies still in flight land
  }
  ok = __syncthreads_and(ok);

  if (ok) {
    // Zero rows >= len of every K and V tile (whole 128-byte rows, so the
    // swizzle does not matter).  2*SPLIT operands x 2 heads x (64 - len) rows.
    const int dead = kChunk - cd.len;
    if (dead > 0) {
      const int rows_total = 2 * SPLIT * kChunkBoxHeads * dead;
      for (int r = tid; r < rows_total * 8; r += kThreads) {
        const int piece = r & 7;           // 16-byte piece of the row
        const int idx = r >> 3;            // which dead row
        const int tile = idx / dead;       // operand part x head tile
        const int row = cd.len + idx % dead;
        uint4* p = reinterpret_cast<uint4*>(smem + tile * kHeadTileBytes + row * 128 + piece * 16);
        *p = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();

  if (ok && tid == 0) {
    tc_fence_after_sync();
    constexpr uint32_t idesc = idesc_bf16_f32(128, 64, /*a MN*/ 1, /*b MN*/ 1);
    for (int hh = 0; hh < kChunkBoxHeads; ++hh) {
      const uint32_t d_tmem = tmem + hh * 64;
      int n = 0;
      for (int kk = 0; kk < kChunk / 16; ++kk) {
        for (int combo = 0; combo < (SPLIT == 2 ? 3 : 1); ++combo) {
          const int pa = (combo == 2) ? 1 : 0;   // hi*hi, hi*lo, lo*hi
          const int pb = (combo == 1) ? 1 : 0;
          const uint64_t a = smem_desc_sw128(base + L::kK + pa * kOperandBytes + kk * 2048,
                                             kHeadTileBytes, 1024);
          const uint64_t b = smem_desc_sw128(
              base + L::kV + pb * kOperandBytes + hh * kHeadTileBytes + kk * 2048,
              kHeadTileBytes, 1024);
          mma_bf16(d_tmem, a, b, idesc, n > 0 ? 1u : 0u);
          ++n;
        }
      }
    }
    mma_commit(bar_mma);
  }

  if (ok) {
    bool done = mbar_wait_bounded(bar_mma, 0, kWaitLimitNs);
    if (!done) {
      atomicOr(err, kErrTimeoutMma);
      mbar_wait_bounded(bar_mma, 0, kWaitLimitNs);
    }
    tc_fence_after_sync();
    // Warp w reads TMEM lanes 32w .. 32w+31.  Lanes 0..63 hold K_h0^T V_h0
    // (columns 0..63), lanes 64..127 hold K_h1^T V_h1 (columns 64..127).
    const int hh = warp >> 1;
    const int h = h0 + hh;
    const int i = tid - hh * 64;   // key-dimension row of the state
    uint32_t r0[32], r1[32];
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16) + hh * 64;
    tmem_ld_32cols(taddr, r0);
    tmem_ld_32cols(taddr + 32, r1);
    tmem_ld_wait();
    if (done && h < H) {
      float4* dst = reinterpret_cast<float4*>(
          ws + ((static_cast<int64_t>(chunk) * H + h) * kHeadDim + i) * kHeadDim);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        dst[c] = make_float4(__uint_as_float(r0[4 * c]), __uint_as_float(r0[4 * c + 1]),
                             __uint_as_float(r0[4 * c + 2]), __uint_as_float(r0[4 * c + 3]));
#pragma unroll
      for (int c = 0; c < 8; ++c)
        dst[8 + c] = make_float4(__uint_as_float(r1[4 * c]), __uint_as_float(r1[4 * c + 1]),
                                 __uint_as_float(r1[4 * c + 2]), __uint_as_float(r1[4 * c + 3]));
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_chunk_state(bool split, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                               const ChunkDesc* chunks, int n_chunks, int H, float* ws,
                               unsigned* err, cudaStream_t stream, bool pdl) {
  if (n_chunks <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_chunks, (H + kChunkBoxHeads - 1) / kChunkBoxHeads);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (split) {
    auto kern = chunk_state_kernel<2>;
    cfg.dynamicSmemBytes = ChunkSmem<2>::kRequest;
    static std::atomic<uint64_t> done{0};
    cudaError_t e = set_smem_limit_once(kern, static_cast<uint32_t>(cfg.dynamicSmemBytes), done);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, kern, tm_k[0], tm_k[1], tm_v[0], tm_v[1], chunks, H, ws, err);
  }
  auto kern = chunk_state_kernel<1>;
  cfg.dynamicSmemBytes = ChunkSmem<1>::kRequest;
  static std::atomic<uint64_t> done{0};
  cudaError_t e = set_smem_limit_once(kern, static_cast<uint32_t>(cfg.dynamicSmemBytes), done);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, kern, tm_k[0], tm_k[0], tm_v[0], tm_v[0], chunks, H, ws, err);
}

}  // namespace spanla
