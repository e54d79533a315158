// Span-state kernel (bf16 inputs): the local state sum_t k_t v_t^T of every
// span, i.e. of a run of consecutive 64-row chunks of one segment.
//
// "Serving 0.88M TPS from Two RTXs and Mac Minis", section "Kernels": the
// per-chunk 64x64 products K_c^T V_c of the chunked form, here summed over the
// chunks of a span inside the tensor cores' fp32 accumulator, so that the scan
// that follows (one scan for every view of the pass) moves one state per span
// instead of one per chunk.
//
// One CTA (128 threads) handles one span for two adjacent heads h0, h0+1.  A
// three-stage TMA ring brings K and V of both heads in 64-row chunks
// ([head][64 rows][64 d] bf16, 128-byte swizzle).  Both operands of K^T V are
// MN-major (the contraction runs over tokens, the row dimension):
//   A (M = 128) = [K_h0 | K_h1]^T, B (N = 64) = V_h,
// so TMEM columns 64h..64h+63 accumulate [K_h0^T V_h ; K_h1^T V_h] and lanes
// 64h..64h+63 of them hold the wanted K_h^T V_h.  Rows of the last chunk past
// the span's end are zeroed in shared memory before its MMAs.
#include "spanla_internal.h"
#include "tc_ptx.cuh"

namespace spanla {
namespace {

constexpr int kThreads = 128;
constexpr int kStages = 3;
constexpr uint32_t kHeadTileBytes = kChunk * 128;                     // 64 rows x 128 B
constexpr uint32_t kOperandBytes = kChunkBoxHeads * kHeadTileBytes;   // 16 KiB (2 heads)
constexpr uint32_t kStageBytes = 2 * kOperandBytes;                   // K + V
constexpr uint32_t kTmemCols = 128;

struct SpanSmem {
  static constexpr uint32_t kStage0 = 0;
  static constexpr uint32_t kBarFull = kStages * kStageBytes;
  static constexpr uint32_t kBarEmpty = kBarFull + 8 * kStages;
  static constexpr uint32_t kBarDone = kBarEmpty + 8 * kStages;
  static constexpr uint32_t kTmemSlot = kBarDone + 8;
  static constexpr uint32_t kBytes = kTmemSlot + 8;
  static constexpr uint32_t kRequest = kBytes + 1024;
};

__global__ void __launch_bounds__(kThreads)
span_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const SpanDesc* __restrict__ spans, int H, float* __restrict__ ws,
                  unsigned* __restrict__ err) {
  using L = SpanSmem;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  // One CTA per (span, head pair); head pairs vary fastest, so the CTAs
  // reading the same rows run together.
  const int pairs = (H + kChunkBoxHeads - 1) / kChunkBoxHeads;
  const int span = blockIdx.x / pairs;
  const int h0 = (blockIdx.x % pairs) * kChunkBoxHeads;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(base + L::kBarFull + 8 * s, 1);
      mbar_init(base + L::kBarEmpty + 8 * s, 1);
    }
    mbar_init(base + L::kBarDone, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  griddep_wait();   // descriptors come from a copy earlier in the stream
  const SpanDesc sd = spans[span];
  const int n_chunks = (sd.len + kChunk - 1) / kChunk;
  const int tail = sd.len - (n_chunks - 1) * kChunk;   // rows of the last chunk

  auto issue_load = [&](int c) {
    const int s = c % kStages;
    const uint32_t st = base + L::kStage0 + s * kStageBytes;
    const uint32_t full = base + L::kBarFull + 8 * s;
    mbar_arrive_expect_tx(full, kStageBytes);
    tma_load_3d(st, &tm_k, full, 0, sd.row0 + c * kChunk, h0);
    tma_load_3d(st + kOperandBytes, &tm_v, full, 0, sd.row0 + c * kChunk, h0);
  };

  // Thread 0 issues every load and MMA.  `issued` / `consumed` count chunks
  // whose loads were issued / whose MMAs were issued (thread 0 only).
  bool ok = true;
  int issued = 0, consumed = 0;
  if (tid == 0)
    for (; issued < n_chunks && issued < kStages; ++issued) issue_load(issued);

  constexpr uint32_t idesc = idesc_bf16_f32(128, 64, /*a MN*/ 1, /*b MN*/ 1);
  for (int c = 0; c < n_chunks; ++c) {
    const int s = c % kStages;
    const uint32_t ph = (c / kStages) & 1;
    const uint32_t st = base + L::kStage0 + s * kStageBytes;
    const uint32_t full = base + L::kBarFull + 8 * s;
    const uint32_t empty = base + L::kBarEmpty + 8 * s;
    const bool partial = (c == n_chunks - 1) && tail < kChunk;
    if (partial) {
      // Only the last chunk can be partial.  Thread 0 reaches this barrier
      // after issuing the MMAs of every earlier chunk, so the stage's barrier
      // is now in this chunk's phase.  Every thread then helps zero rows
      // >= tail of the 4 head tiles of K and V.
      ok = __syncthreads_and(ok);
      if (ok) {
        const bool got = mbar_wait_bounded(full, ph, kWaitLimitNs);
        if (got) {
          const int dead = kChunk - tail;
          uint8_t* stage = smem + (st - base);
          for (int r = tid; r < 4 * dead * 8; r += kThreads) {
            const int piece = r & 7, idx = r >> 3;
            const int tile = idx / dead, row = tail + idx % dead;
            *reinterpret_cast<uint4*>(stage + tile * kHeadTileBytes + row * 128 + piece * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        } else {
          atomicOr(err, kErrTimeoutTma);
        }
        ok = __syncthreads_and(got);
      }
    }
    if (tid == 0 && ok) {
      if (!partial && !mbar_wait_bounded(full, ph, kWaitLimitNs)) {
        atomicOr(err, kErrTimeoutTma);
        ok = false;
      }
      if (ok) {
        tc_fence_after_sync();
        for (int hh = 0; hh < kChunkBoxHeads; ++hh) {
          for (int kk = 0; kk < kChunk / 16; ++kk) {
            const uint64_t a = smem_desc_sw128(st + kk * 2048, kHeadTileBytes, 1024);
            const uint64_t b = smem_desc_sw128(st + kOperandBytes + hh * kHeadTileBytes + kk * 2048,
                                               kHeadTileBytes, 1024);
            mma_bf16(tmem + hh * 64, a, b, idesc, (c > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(empty);
        consumed = c + 1;
        if (issued < n_chunks) {
          // The stage is reloaded once the MMAs reading it have completed.
          if (!mbar_wait_bounded(empty, ph, kWaitLimitNs)) {
            atomicOr(err, kErrTimeoutMma);
            ok = false;
          } else {
            issue_load(issued++);
          }
        }
      }
    }
  }
  if (tid == 0) {
    if (ok) {
      mma_commit(base + L::kBarDone);
    } else {
      // Give up: let the loads still in flight land (bounded) before the
      // CTA's shared memory is released.
      for (int c = consumed; c < issued; ++c)
        mbar_wait_bounded(base + L::kBarFull + 8 * (c % kStages), (c / kStages) & 1, 1000000ull);
    }
  }
  griddep_launch_dependents();
  ok = __syncthreads_and(ok);

  if (ok) {
    const bool done = mbar_wait_bounded(base + L::kBarDone, 0, kWaitLimitNs);
    if (!done) atomicOr(err, kErrTimeoutMma);
    tc_fence_after_sync();
    const int hh = warp >> 1;
    const int h = h0 + hh;
    const int i = tid - hh * 64;
    uint32_t r0[32], r1[32];
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16) + hh * 64;
    tmem_ld_32cols(taddr, r0);
    tmem_ld_32cols(taddr + 32, r1);
    tmem_ld_wait();
    if (done && h < H) {
      float4* dst = reinterpret_cast<float4*>(
          ws + ((static_cast<int64_t>(span) * H + h) * kHeadDim + i) * kHeadDim);
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

cudaError_t launch_span_state(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                              const SpanDesc* spans, int n_spans, int H, float* ws,
                              unsigned* err, cudaStream_t stream) {
  if (n_spans <= 0) return cudaSuccess;
  const int64_t ctas = static_cast<int64_t>(n_spans) * ((H + kChunkBoxHeads - 1) / kChunkBoxHeads);
  if (ctas > INT32_MAX) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(ctas));
  const uint32_t bytes = SpanSmem::kRequest;
  cudaError_t e =
      cudaFuncSetAttribute(span_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  span_state_kernel<<<grid, kThreads, bytes, stream>>>(tm_k[0], tm_v[0], spans, H, ws, err);
  return cudaGetLastError();
}

}  // namespace spanla
