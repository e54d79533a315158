// Span-output kernel (bf16 inputs): the output of every view row and every
// branch row, carrying the state across the tiles of a span.
//
// "Serving 0.88M TPS from Two RTXs and Mac Minis", section "Kernels" (each
// 64-token chunk: a masked Q K^T times V inside the chunk plus Q times the
// state entering it; shared branch passes with the small kernels fused) and
// section "The Workload" (branches attend to the view, not to each other).
//
// Work unit = (item, head).  An item is a span (up to G consecutive 128-row
// tiles of a view or of a long branch) or one tile of packed short branches
// of one parent.  With S the state entering a tile (the item's start state
// stateA[a] + stateB[b] for its first tile: the scan prefix and/or the
// parent view's final state -- the branch fork), every row i of the tile gets
//
//     o_i = sum_{start(i) <= j <= i} (q_i . k_j) v_j  +  S^T q_i ,
//
// and the next tile of the item starts from S + K^T V of this one.
//
// Persistent CTAs (one per SM) walk a host-built list of tiles.  6 warps:
//   warp 0     producer: Q, K, V tiles by TMA and, at an item's first tile,
//              its fp32 start states by bulk copy, into a two-stage ring
//   warp 1     MMA issuer (one lane; the warp zeroes partial-tile K/V rows),
//              two TMEM accumulator buffers b = tile & 1:
//                P_b  = Q K^T              M128 N128 K64
//                O_b  = Q S_hi + Q S_lo    M128 N64  K64
//                dS (+)= K^T V             M128 N64  K128
//                O_b += P V                M128 N64  K128
//              so P of the next tile is computed while the epilogue is still
//              storing O of this one
//   warps 2-5  epilogue, one tile row per thread (TMEM lane): P -> masked
//              bf16 A operand; S + dS -> bf16 high/low B operand of the next
//              tile; O -> global.
// K^T V uses both tiles MN-major with M = 128: the second 64-wide M atom is the
// V tile, so TMEM lanes 64..127 of dS are unused.
#include "spanla_internal.h"
#include "tc_ptx.cuh"

namespace spanla {
namespace {

constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr uint32_t kRowTileBytes = kTileRows * 128;        // 128 rows x 128 B
constexpr uint32_t kStateBytes = kStateFloats * 4;         // fp32 64 x 64
constexpr uint32_t kStageBytes = 3 * kRowTileBytes + 2 * kStateBytes;   // Q K V SA SB
constexpr uint32_t kStateTileBytes = kHeadDim * 128;       // 64 rows x 128 B (bf16)
constexpr uint32_t kTmemCols = 512;
// TMEM columns: buffer b holds P at kColP<b> (128) and O at kColO<b> (64).
constexpr uint32_t kColP0 = 0, kColO0 = 128, kColS = 192, kColP1 = 256, kColO1 = 384;

struct OutSmem {
  static constexpr uint32_t kStage0 = 0;
  static constexpr uint32_t kQ = 0, kK = kRowTileBytes, kV = 2 * kRowTileBytes,
                            kSA = 3 * kRowTileBytes, kSB = 3 * kRowTileBytes + kStateBytes;
  static constexpr uint32_t kS = kStages * kStageBytes;          // S hi, S lo (bf16)
  static constexpr uint32_t kP = kS + 2 * kStateTileBytes;       // [2 blocks][128][64] bf16
  static constexpr uint32_t kBar = kP + 2 * kRowTileBytes;
  // barrier slots (8 bytes each)
  static constexpr int kFull = 0, kEmpty = 2, kPReady = 4, kOReady = 6, kTmemFree = 8,
                       kSAccReady = 10, kPSmem = 11, kSSmem = 12, kNumBars = 13;
  static constexpr uint32_t kTmemSlot = kBar + 8 * kNumBars;
  static constexpr uint32_t kBytes = kTmemSlot + 8;
  static constexpr uint32_t kRequest = kBytes + 1024;
};
static_assert(OutSmem::kRequest <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ bool wait_or_flag(uint32_t bar, uint32_t parity, unsigned* err,
                                             unsigned code) {
  if (mbar_wait_bounded(bar, parity, kWaitLimitNs)) return true;
  atomicOr(err, code);
  return false;
}

__device__ __forceinline__ WorkTile load_tile(const WorkTile* p) {
  WorkTile t;
  const uint4* src = reinterpret_cast<const uint4*>(p);
  uint4* dst = reinterpret_cast<uint4*>(&t);
  dst[0] = __ldg(src);
  dst[1] = __ldg(src + 1);
  dst[2] = __ldg(src + 2);
  return t;
}

// Write 64 state values of row d as bf16 high / low parts into the MN-major
// S operand ([d][64 e], 128-byte swizzle).
__device__ __forceinline__ void stage_state_row(uint8_t* s_op, int d, const float* x) {
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float h0, l0, h1, l1;
      split_bf16(x[8 * g + 2 * u], h0, l0);
      split_bf16(x[8 * g + 2 * u + 1], h1, l1);
      hi[u] = pack_bf16x2(h0, h1);
      lo[u] = pack_bf16x2(l0, l1);
    }
    const uint32_t off = sw128_offset(d, 8 * g);
    *reinterpret_cast<uint4*>(s_op + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(s_op + kStateTileBytes + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
span_output_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const WorkTile* __restrict__ work,
                   const int32_t* __restrict__ cta_begin, const uint8_t* __restrict__ bounds,
                   const float* __restrict__ stateA, const float* __restrict__ stateB,
                   __nv_bfloat16* __restrict__ out, int H, unsigned* __restrict__ err) {
  using L = OutSmem;
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
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kFull + s), 1);
      mbar_init(bar(L::kEmpty + s), 1);
      mbar_init(bar(L::kPReady + s), 1);
      mbar_init(bar(L::kOReady + s), 1);
      mbar_init(bar(L::kTmemFree + s), 128);
    }
    mbar_init(bar(L::kSAccReady), 1);
    mbar_init(bar(L::kPSmem), 128);
    mbar_init(bar(L::kSSmem), 128);
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  griddep_wait();   // states from the scan, schedule from the descriptor copy
  const int i_begin = cta_begin[blockIdx.x];
  const int n = cta_begin[blockIdx.x + 1] - i_begin;
  const WorkTile* list = work + i_begin;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      int i = 0;
      WorkTile nxt = n > 0 ? load_tile(list) : WorkTile{};
      for (; i < n; ++i) {
        const WorkTile r = nxt;
        if (i + 1 < n) nxt = load_tile(list + i + 1);
        const int s = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!wait_or_flag(bar(L::kEmpty + s), ph ^ 1, err, kErrTimeoutMma)) { ok = false; break; }
        const uint32_t st = base + L::kStage0 + s * kStageBytes;
        const bool first = r.flags & kTileFirst;
        const bool ld_a = first && r.stateA >= 0, ld_b = first && r.stateB >= 0;
        mbar_arrive_expect_tx(bar(L::kFull + s), 3 * kRowTileBytes + (ld_a ? kStateBytes : 0) +
                                                      (ld_b ? kStateBytes : 0));
        tma_load_3d(st + L::kQ, &tm_q, bar(L::kFull + s), 0, r.row0, r.head);
        tma_load_3d(st + L::kK, &tm_k, bar(L::kFull + s), 0, r.row0, r.head);
        tma_load_3d(st + L::kV, &tm_v, bar(L::kFull + s), 0, r.row0, r.head);
        if (ld_a)
          bulk_copy_g2s(st + L::kSA, stateA + (static_cast<int64_t>(r.stateA) * H + r.head) * kStateFloats,
                        kStateBytes, bar(L::kFull + s));
        if (ld_b)
          bulk_copy_g2s(st + L::kSB, stateB + (static_cast<int64_t>(r.stateB) * H + r.head) * kStateFloats,
                        kStateBytes, bar(L::kFull + s));
      }
      // Wait (bounded) for the last loads to land before the CTA can exit.
      for (int u = (i > kStages ? i - kStages : 0); u < i; ++u)
        mbar_wait_bounded(bar(L::kFull + (u & 1)), (u >> 1) & 1, ok ? kWaitLimitNs : 1000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    bool ok = true;
    constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, 0, 0);
    constexpr uint32_t id_n64_b_mn = idesc_bf16_f32(128, 64, 0, 1);
    constexpr uint32_t id_kv = idesc_bf16_f32(128, 64, 1, 1);
    WorkTile nxt = n > 0 ? load_tile(list) : WorkTile{};
    for (int i = 0; i < n && ok; ++i) {
      const WorkTile r = nxt;
      if (i + 1 < n) nxt = load_tile(list + i + 1);
      const int s = i & 1, b = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      const uint32_t st = base + L::kStage0 + s * kStageBytes;
      const uint32_t sq = st + L::kQ, sk = st + L::kK, sv = st + L::kV;
      const uint32_t colP = b ? kColP1 : kColP0, colO = b ? kColO1 : kColO0;
      const bool first = r.flags & kTileFirst, last = r.flags & kTileLast;
      const bool has_state = !first || (r.flags & kTileHasInit);

      ok = __all_sync(0xffffffffu, wait_or_flag(bar(L::kFull + s), ph, err, kErrTimeoutTma));
      if (!ok) break;
      if (r.nrows < kTileRows) {
        // K and V rows past the tile may hold anything, even NaN; zero them so
        // masked P entries and the state update multiply zeros.
        uint8_t* vrow = smem + (sv - base);
        uint8_t* krow = smem + (sk - base);
        for (int q = r.nrows * 8 + lane; q < kTileRows * 8; q += 32) {
          *reinterpret_cast<uint4*>(vrow + q * 16) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(krow + q * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (i >= 2) ok = wait_or_flag(bar(L::kTmemFree + b), ((i - 2) >> 1) & 1, err, kErrTimeoutMma);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      if (lane == 0) {
        for (int kk = 0; kk < kHeadDim / 16; ++kk)
          mma_bf16(tmem + colP, smem_desc_sw128(sq + kk * 32, 16, 1024),
                   smem_desc_sw128(sk + kk * 32, 16, 1024), id_qk, kk > 0);
        mma_commit(bar(L::kPReady + b));
      }
      __syncwarp();
      // S of this tile (staged by the epilogue) -> O_b = Q S, and the state
      // update for the next tile of the item.
      ok = __all_sync(0xffffffffu, wait_or_flag(bar(L::kSSmem), i & 1, err, kErrTimeoutMma));
      if (!ok) break;
      tc_fence_after_sync();
      if (lane == 0) {
        if (has_state) {
          int m = 0;
          for (int kk = 0; kk < kHeadDim / 16; ++kk)
            for (int part = 0; part < 2; ++part, ++m)
              mma_bf16(tmem + colO, smem_desc_sw128(sq + kk * 32, 16, 1024),
                       smem_desc_sw128(base + L::kS + part * kStateTileBytes + kk * 2048,
                                       kStateTileBytes, 1024),
                       id_n64_b_mn, m > 0);
        }
        if (!last) {
          for (int kk = 0; kk < kTileRows / 16; ++kk)
            mma_bf16(tmem + kColS, smem_desc_sw128(sk + kk * 2048, kRowTileBytes, 1024),
                     smem_desc_sw128(sv + kk * 2048, kRowTileBytes, 1024), id_kv,
                     (!first || kk > 0) ? 1u : 0u);
          mma_commit(bar(L::kSAccReady));
        }
      }
      __syncwarp();
      ok = __all_sync(0xffffffffu, wait_or_flag(bar(L::kPSmem), i & 1, err, kErrTimeoutMma));
      if (!ok) break;
      tc_fence_after_sync();
      if (lane == 0) {
        for (int kk = 0; kk < kTileRows / 16; ++kk)
          mma_bf16(tmem + colO,
                   smem_desc_sw128(base + L::kP + (kk >> 2) * kRowTileBytes + (kk & 3) * 32, 16, 1024),
                   smem_desc_sw128(sv + kk * 2048, kRowTileBytes, 1024), id_n64_b_mn,
                   (has_state || kk > 0) ? 1u : 0u);
        mma_commit(bar(L::kOReady + b));
        mma_commit(bar(L::kEmpty + s));
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;          // tile row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const bool state_rows = quarter < 2;          // lanes 0..63 hold state rows
    uint32_t sacc = 0;
    bool ok = true;
    float s_init[64];
    WorkTile nxt = n > 0 ? load_tile(list) : WorkTile{};
    for (int i = 0; i < n && ok; ++i) {
      const WorkTile r = nxt;
      if (i + 1 < n) nxt = load_tile(list + i + 1);
      const int s = i & 1, b = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      const uint32_t colP = b ? kColP1 : kColP0, colO = b ? kColO1 : kColO0;
      const bool first = r.flags & kTileFirst, last = r.flags & kTileLast;

      if (first) {
        // The item's start state (landed with the stage) -> S operand.
        const bool has_init = r.flags & kTileHasInit;
        if (has_init) {
          ok = __all_sync(0xffffffffu, wait_or_flag(bar(L::kFull + s), ph, err, kErrTimeoutTma));
          if (!ok) break;
        }
        if (state_rows) {
          const uint8_t* st = smem + L::kStage0 + s * kStageBytes;
#pragma unroll
          for (int e = 0; e < 64; ++e) s_init[e] = 0.f;
          if (r.stateA >= 0) {
            const float4* a = reinterpret_cast<const float4*>(st + L::kSA) + row * 16;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float4 x = a[c];
              s_init[4 * c] += x.x; s_init[4 * c + 1] += x.y;
              s_init[4 * c + 2] += x.z; s_init[4 * c + 3] += x.w;
            }
          }
          if (r.stateB >= 0) {
            const float4* bb = reinterpret_cast<const float4*>(st + L::kSB) + row * 16;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float4 x = bb[c];
              s_init[4 * c] += x.x; s_init[4 * c + 1] += x.y;
              s_init[4 * c + 2] += x.z; s_init[4 * c + 3] += x.w;
            }
          }
          if (has_init) stage_state_row(smem + L::kS, row, s_init);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(L::kSSmem));
      }

      // Segment start of this row inside the tile.
      int seg_start = 0;
      if (r.nbound > 1) {
        const int nb = r.nbound < kInlineBounds ? r.nbound : kInlineBounds;
        for (int q = 1; q < nb; ++q)
          if (r.inl[q] <= row) seg_start = r.inl[q];
        for (int q = kInlineBounds; q < r.nbound; ++q) {
          const int sb = bounds[r.bound0 + q];
          if (sb <= row) seg_start = sb;
        }
      }

      // P row -> mask -> bf16 -> K-major A operand of P V.
      ok = __all_sync(0xffffffffu, wait_or_flag(bar(L::kPReady + b), ph, err, kErrTimeoutMma));
      if (!ok) break;
      tc_fence_after_sync();
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t r0[32], r1[32];
        tmem_ld_32cols(tmem + lane_base + colP + half * 64, r0);
        tmem_ld_32cols(tmem + lane_base + colP + half * 64 + 32, r1);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const int j0 = half * 64 + g * 8;
          uint32_t pk[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int jj = j0 + 2 * u;
            const int ci = (g & 3) * 8 + 2 * u;
            float p0 = __uint_as_float(g < 4 ? r0[ci] : r1[ci]);
            float p1 = __uint_as_float(g < 4 ? r0[ci + 1] : r1[ci + 1]);
            p0 = (jj >= seg_start && jj <= row && row < r.nrows) ? p0 : 0.f;
            p1 = (jj + 1 >= seg_start && jj + 1 <= row && row < r.nrows) ? p1 : 0.f;
            pk[u] = pack_bf16x2(p0, p1);
          }
          const uint32_t off = half * kRowTileBytes + sw128_offset(row, g * 8);
          *reinterpret_cast<uint4*>(smem + L::kP + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kPSmem));

      if (!last) {
        // Next tile's state S + dS -> S operand.
        ok = __all_sync(0xffffffffu, wait_or_flag(bar(L::kSAccReady), sacc & 1, err, kErrTimeoutMma));
        ++sacc;
        if (!ok) break;
        tc_fence_after_sync();
        if (state_rows) {
          uint32_t r0[32], r1[32];
          tmem_ld_32cols(tmem + lane_base + kColS, r0);
          tmem_ld_32cols(tmem + lane_base + kColS + 32, r1);
          tmem_ld_wait();
          float x[64];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = s_init[e] + __uint_as_float(r0[e]);
            x[e + 32] = s_init[e + 32] + __uint_as_float(r1[e]);
          }
          stage_state_row(smem + L::kS, row, x);
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        mbar_arrive(bar(L::kSSmem));
      }

      // O row -> global.
      ok = __all_sync(0xffffffffu, wait_or_flag(bar(L::kOReady + b), ph, err, kErrTimeoutMma));
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t r0[32], r1[32];
      tmem_ld_32cols(tmem + lane_base + colO, r0);
      tmem_ld_32cols(tmem + lane_base + colO + 32, r1);
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kTmemFree + b));
      if (row < r.nrows) {
        uint4* dst = reinterpret_cast<uint4*>(
            out + ((static_cast<int64_t>(r.row0) + row) * H + r.head) * kHeadDim);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          dst[c] = make_uint4(pack_bf16x2(__uint_as_float(r0[8 * c]), __uint_as_float(r0[8 * c + 1])),
                              pack_bf16x2(__uint_as_float(r0[8 * c + 2]), __uint_as_float(r0[8 * c + 3])),
                              pack_bf16x2(__uint_as_float(r0[8 * c + 4]), __uint_as_float(r0[8 * c + 5])),
                              pack_bf16x2(__uint_as_float(r0[8 * c + 6]), __uint_as_float(r0[8 * c + 7])));
#pragma unroll
        for (int c = 0; c < 4; ++c)
          dst[4 + c] = make_uint4(pack_bf16x2(__uint_as_float(r1[8 * c]), __uint_as_float(r1[8 * c + 1])),
                                  pack_bf16x2(__uint_as_float(r1[8 * c + 2]), __uint_as_float(r1[8 * c + 3])),
                                  pack_bf16x2(__uint_as_float(r1[8 * c + 4]), __uint_as_float(r1[8 * c + 5])),
                                  pack_bf16x2(__uint_as_float(r1[8 * c + 6]), __uint_as_float(r1[8 * c + 7])));
      }
    }
  }

  griddep_launch_dependents();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_span_output(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                               const CUtensorMap* tm_v, const WorkTile* work,
                               const int32_t* cta_begin, int grid, const uint8_t* bounds,
                               const float* stateA, const float* stateB, void* out, int H,
                               unsigned* err, cudaStream_t stream, bool pdl) {
  if (grid <= 0) return cudaSuccess;
  const uint32_t bytes = OutSmem::kRequest;
  cudaError_t e =
      cudaFuncSetAttribute(span_output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, span_output_kernel, tm_q[0], tm_k[0], tm_v[0], work, cta_begin,
                            bounds, stateA, stateB, static_cast<__nv_bfloat16*>(out), H, err);
}

}  // namespace spanla
