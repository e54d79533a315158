// Span-state kernel (bf16 inputs): the local state sum_t k_t v_t^T of every
// piece, i.e. of a run of consecutive rows of one segment-head.
//
// "Serving 0.88M TPS from Two RTXs and Mac Minis", section "Kernels": the
// per-chunk 64x64 products K_c^T V_c of the chunked form, here summed over the
// chunks of a piece inside the tensor cores' fp32 accumulator, so that the
// scan that follows (one scan for every view of the pass) moves one state per
// piece instead of one per chunk.
//
// Persistent CTAs (one per SM) walk their own list of pieces (the host deals
// the pieces to CTAs longest first onto the least-loaded CTA).  4 warps:
//   warp 2     producer: K and V of one head, 256 rows (four chunks) at a
//              time ([256 rows][64 d] bf16, 128-byte swizzle; 32 KB boxes
//              stream faster than 16 KB ones), into a three-stage ring,
//              running ahead across units.
//   warp 3     MMA issuer: per 256 rows 16 MMAs  acc (+)= K^T V  with both
//              operands MN-major (the contraction runs over tokens): A (M =
//              128) = [K | V]^T -- the V tile is the second 64-wide M atom and
//              only TMEM lanes 0..63 (K^T V) are kept -- and B (N = 64) = V.
//              Two TMEM accumulators alternate between units.  The warp
//              zeroes rows past a segment's end in a partial last chunk.
//   warps 0-1  epilogue: TMEM lanes 0..63 (state rows) -> fp32 state slot.
#include "spanla_internal.h"
#include "tc_ptx.cuh"

namespace spanla {
namespace {

constexpr int kThreads = 128;
constexpr int kStages = 3;
constexpr int kRows = 4 * kChunk;                        // rows per stage
constexpr uint32_t kTileBytes = kRows * 128;             // 128 rows x 128 B (one head)
constexpr uint32_t kStageBytes = 2 * kTileBytes;         // K, V
constexpr uint32_t kTmemCols = 128;                      // two 64-column accumulators
constexpr int kDescSlots = 128;                          // piece records staged in shared memory

struct SpanSmem {
  static constexpr uint32_t kStage0 = 0;
  static constexpr uint32_t kBar = kStages * kStageBytes;
  static constexpr int kFull = 0, kEmpty = kStages, kAccReady = 2 * kStages,
                       kAccFree = 2 * kStages + 2, kNumBars = 2 * kStages + 4;
  static constexpr uint32_t kTmemSlot = kBar + 8 * kNumBars;
  static constexpr uint32_t kDesc = kTmemSlot + 8;               // this CTA's span records
  static constexpr uint32_t kBytes = kDesc + kDescSlots * sizeof(SpanDesc);
  static constexpr uint32_t kRequest = kBytes + 1024;
};

__device__ __forceinline__ bool wait_or_flag(uint32_t bar, uint32_t parity, unsigned* err,
                                             unsigned code) {
  if (mbar_wait_bounded(bar, parity, kWaitLimitNs)) return true;
  atomicOr(err, code);
  return false;
}

__global__ void __launch_bounds__(kThreads, 1)
span_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const SpanDesc* __restrict__ spans, const int32_t* __restrict__ span_begin,
                  float* __restrict__ ws, const uint8_t* __restrict__ prefetch, uint32_t prefetch_bytes,
                  unsigned* __restrict__ err) {
  using L = SpanSmem;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  auto bar = [&](int slot) { return base + L::kBar + 8u * slot; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(L::kFull + s), 1);
      mbar_init(bar(L::kEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(L::kAccReady + b), 1);
      mbar_init(bar(L::kAccFree + b), 64);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  griddep_wait();   // descriptors come from a copy earlier in the stream
  // The scan may be scheduled now: it waits for this grid's completion itself.
  griddep_launch_dependents();
  // The pass's descriptor block (the later kernels' schedules) into L2, a
  // slice per CTA, so that their first reads do not wait on DRAM.
  if (tid == 0 && prefetch_bytes > 0) {
    const uint32_t chunk = ((prefetch_bytes + gridDim.x - 1) / gridDim.x + 15u) & ~15u;
    const uint32_t lo = blockIdx.x * chunk;
    if (lo < prefetch_bytes) bulk_prefetch_l2(prefetch + lo, min(chunk, prefetch_bytes - lo));
  }
  const int u_begin = span_begin[blockIdx.x];
  const int n_units = span_begin[blockIdx.x + 1] - u_begin;
  const SpanDesc* list = spans + u_begin;
  // Stage this CTA's first piece records in shared memory, all loads in
  // flight at once, so the producer does not wait on one per piece.
  SpanDesc* sdesc = reinterpret_cast<SpanDesc*>(smem + L::kDesc);
  for (int j = tid; j < kDescSlots && j < n_units; j += kThreads) sdesc[j] = list[j];
  auto span_of = [&](int j) { return j < kDescSlots ? sdesc[j] : list[j]; };
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 2) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int c = 0;   // running chunk count (ring position)
      bool ok = true;
      for (int j = 0; j < n_units && ok; ++j) {
        const SpanDesc sd = span_of(j);
        const int h = sd.head;
        const int n_chunks = (sd.len + kRows - 1) / kRows;
        for (int q = 0; q < n_chunks; ++q, ++c) {
          const int s = c % kStages;
          if (!wait_or_flag(bar(L::kEmpty + s), ((c / kStages) & 1) ^ 1, err, kErrTimeoutMma)) {
            ok = false;
            break;
          }
          const uint32_t st = base + L::kStage0 + s * kStageBytes;
          mbar_arrive_expect_tx(bar(L::kFull + s), kStageBytes);
          tma_load_3d(st, &tm_k, bar(L::kFull + s), 0, sd.row0 + q * kRows, h);
          tma_load_3d(st + kTileBytes, &tm_v, bar(L::kFull + s), 0, sd.row0 + q * kRows, h);
        }
      }
      // Let the last loads land (bounded) before the CTA can exit.
      for (int u = (c > kStages ? c - kStages : 0); u < c; ++u)
        mbar_wait_bounded(bar(L::kFull + u % kStages), (u / kStages) & 1, ok ? kWaitLimitNs : 1000000ull);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(128, 64, /*a MN*/ 1, /*b MN*/ 1);
    int c = 0;   // running chunk count
    bool ok = true;
    for (int k = 0; k < n_units && ok; ++k) {
      const SpanDesc sd = span_of(k);
      const int n_chunks = (sd.len + kRows - 1) / kRows;
      const int b = k & 1;
      if (k >= 2) ok = wait_or_flag(bar(L::kAccFree + b), ((k - 2) >> 1) & 1, err, kErrTimeoutMma);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after_sync();
      for (int j = 0; j < n_chunks; ++j, ++c) {
        const int s = c % kStages;
        ok = __all_sync(0xffffffffu, wait_or_flag(bar(L::kFull + s), (c / kStages) & 1, err, kErrTimeoutTma));
        if (!ok) break;
        const uint32_t st = base + L::kStage0 + s * kStageBytes;
        const int rows = sd.len - j * kRows;
        if (rows < kRows) {
          // Rows past the span's end belong to other segments: zero them in K and V.
          uint8_t* kt = smem + (st - base);
          for (int q = rows * 8 + lane; q < kRows * 8; q += 32) {
            *reinterpret_cast<uint4*>(kt + q * 16) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(kt + kTileBytes + q * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        tc_fence_after_sync();
        if (lane == 0) {
          for (int kk = 0; kk < kRows / 16; ++kk)
            mma_bf16(tmem + b * 64, smem_desc_sw128(st + kk * 2048, kTileBytes, 1024),
                     smem_desc_sw128(st + kTileBytes + kk * 2048, kTileBytes, 1024), idesc,
                     (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(L::kEmpty + s));
          if (j + 1 == n_chunks) mma_commit(bar(L::kAccReady + b));
        }
        __syncwarp();
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 0, 1)
    const int d = warp * 32 + lane;   // state row = TMEM lane (0..63)
    for (int k = 0; k < n_units; ++k) {
      const int b = k & 1;
      const int slot = span_of(k).slot;
      if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kAccReady + b), (k >> 1) & 1, err, kErrTimeoutMma)))
        break;
      tc_fence_after_sync();
      uint32_t r0[32], r1[32];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16) + b * 64;
      tmem_ld_32cols(taddr, r0);
      tmem_ld_32cols(taddr + 32, r1);
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kAccFree + b));
      float4* dst = reinterpret_cast<float4*>(ws + (static_cast<int64_t>(slot) * kHeadDim + d) * kHeadDim);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[q] = make_float4(__uint_as_float(r0[4 * q]), __uint_as_float(r0[4 * q + 1]),
                             __uint_as_float(r0[4 * q + 2]), __uint_as_float(r0[4 * q + 3]));
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[8 + q] = make_float4(__uint_as_float(r1[4 * q]), __uint_as_float(r1[4 * q + 1]),
                                 __uint_as_float(r1[4 * q + 2]), __uint_as_float(r1[4 * q + 3]));
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_span_state(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                              const SpanDesc* spans, const int32_t* span_begin, int grid,
                              float* ws, const void* prefetch, size_t prefetch_bytes, unsigned* err,
                              cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  const uint32_t bytes = SpanSmem::kRequest;
  static std::atomic<uint64_t> done{0};
  cudaError_t e = set_smem_limit_once(span_state_kernel, bytes, done);
  if (e != cudaSuccess) return e;
  span_state_kernel<<<grid, kThreads, bytes, stream>>>(
      tm_k[0], tm_v[0], spans, span_begin, ws, static_cast<const uint8_t*>(prefetch),
      static_cast<uint32_t>(prefetch_bytes & ~static_cast<size_t>(15)), err);
  return cudaGetLastError();
}

}  // namespace spanla
