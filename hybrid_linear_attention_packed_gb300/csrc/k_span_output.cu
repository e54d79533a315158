// Span-output kernel (bf16 inputs): the output of every view row and every
// branch row, carrying the state across the tiles of a piece.
//
// "Serving 0.88M TPS from Two RTXs and Mac Minis", section "Kernels" (each
// 64-token chunk: a masked Q K^T times V inside the chunk plus Q times the
// state entering it; shared branch passes with the small kernels fused) and
// section "The Workload" (branches attend to the view, not to each other).
//
// Each CTA runs one contiguous run of (tile, head) work from a host-built
// list.  A piece is the part of one view-head or long-branch-head inside the
// run; a tile of packed short branches is a piece of its own.  With S the
// state entering a tile (the piece's start state stateA[a] + stateB[b] for
// its first tile: the scan prefix and/or the parent view's final state -- the
// branch fork), every row i of the tile gets
//
//     o_i = sum_{start(i) <= j <= i} (q_i . k_j) v_j  +  S^T q_i ,
//
// and the next tile of the piece starts from S + K^T V of this one.
//
// Software pipelined over consecutive tiles t.  15 warps:
//   warp 0     producer: Q, K, V tiles by TMA into a four-stage ring.
//   warp 1     front issuer (one lane; the warp zeroes partial-tile K/V
//              rows), as soon as tile t has landed:  P(t) = Q K^T  (M128
//              N128 K64) into TMEM buffer t & 1, then, unless t ends its
//              piece, the tile's own state  dS(t) = K^T V  (M128 N64 K128)
//              into TMEM region t & 1.
//   warp 2     O issuer (one lane): once the P conversion has turned P(t)
//              into bf16 in place,  O(t) = P(t) V  (M128 N64 K128, P read
//              from tensor memory), then, with S(t) staged,  O(t) += Q S_hi +
//              Q S_lo  (M128 N64 K64), so that an O buffer is held only from
//              the end of the conversion until the tile's output is read.
//   warps 3-10 P conversion, two warps per TMEM lane quarter, one per
//              64-column half: each thread owns one tile row (TMEM lane) and
//              turns its half of P(t) into the masked bf16 A operand in place
//              in tensor memory -- 64 fp32 columns become 64 bf16 in the half's
//              first 32 columns (P V reads keys 0..63 from columns 0..31 and
//              keys 64..127 from columns 64..95).
//   warps 11-14 state and output, one warp per lane quarter.  They hold the
//              running fp32 state in registers (a 32-column half of one state
//              row per thread); per step t they add dS(t) to it (or load the
//              next piece's start state, fetched a tile ahead), stage S(t+1)
//              as bf16 high / low parts for Q S, and then store O(t).
// No tensor-core work waits on the state warps' arithmetic except Q S, and
// the state chain runs through registers only, so the tensor pipe sees the
// MMAs of consecutive tiles back to back.  K^T V runs with M = 128 and the K
// tile as both 64-wide M atoms, so TMEM lanes 64..127 hold a copy of dS rows
// 0..63: the lower copy is read for columns 0..31, the upper for 32..63.
#include "spanla_internal.h"
#include "tc_ptx.cuh"

namespace spanla {
namespace {

constexpr int kThreads = 480;
constexpr int kGroupWarps = 4;                           // state and output
constexpr int kGroupThreads = 32 * kGroupWarps;
constexpr int kConvWarps = 8;                            // P conversion
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kStages = 4;
constexpr uint32_t kRowTileBytes = kTileRows * 128;        // 128 rows x 128 B
constexpr uint32_t kStageBytes = 3 * kRowTileBytes;       // Q K V
constexpr uint32_t kStateTileBytes = kHeadDim * 128;       // 64 rows x 128 B (bf16)
constexpr uint32_t kSOpBytes = 2 * kStateTileBytes;         // S as bf16 hi + lo
constexpr int kCoordSlots = 64;                              // tile coordinates staged for the producer
constexpr uint32_t kTmemCols = 512;
// TMEM columns: P buffers (128 each), O buffers (64 each), dS regions (64 each).
constexpr uint32_t kColP0 = 0, kColP1 = 128, kColO0 = 256, kColO1 = 320, kColD0 = 384, kColD1 = 448;

struct OutSmem {
  static constexpr uint32_t kStage0 = 0;
  static constexpr uint32_t kQ = 0, kK = kRowTileBytes, kV = 2 * kRowTileBytes;
  static constexpr uint32_t kS = kStages * kStageBytes;          // two S operands (hi, lo)
  static constexpr uint32_t kBar = kS + 2 * kSOpBytes;
  // barrier slots (8 bytes each); the pairs are used by alternate tiles.
  // Empty takes two arrivals per tile: the front issuer's MMAs and the O
  // issuer's MMAs both read the stage.
  static constexpr int kFull = 0, kEmpty = kStages, kPReady = 2 * kStages,
                       kPDone = kPReady + 2, kOReady = kPReady + 4, kOFree = kPReady + 6,
                       kSSmem = kPReady + 8, kDReady = kPReady + 10, kDFree = kPReady + 12,
                       kNumBars = kPReady + 14;
  static constexpr uint32_t kTmemSlot = kBar + 8 * kNumBars;
  static constexpr uint32_t kCoord = kTmemSlot + 8;              // (row0, head) of the first tiles
  static constexpr uint32_t kBytes = kCoord + 8 * kCoordSlots;
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

// Write 32 state values (columns 32*half ..) of row d as bf16 high / low parts
// into the MN-major S operand ([d][64 e], 128-byte swizzle).
__device__ __forceinline__ void stage_state_half_row(uint8_t* s_op, int d, int half, const float* x) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float h0, l0, h1, l1;
      split_bf16(x[8 * g + 2 * u], h0, l0);
      split_bf16(x[8 * g + 2 * u + 1], h1, l1);
      hi[u] = pack_bf16x2(h0, h1);
      lo[u] = pack_bf16x2(l0, l1);
    }
    const uint32_t off = sw128_offset(d, 32 * half + 8 * g);
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
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(L::kFull + s), 1);
      mbar_init(bar(L::kEmpty + s), 2);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(L::kPReady + b), 1);
      mbar_init(bar(L::kPDone + b), kConvThreads);
      mbar_init(bar(L::kOReady + b), 1);
      mbar_init(bar(L::kOFree + b), kGroupThreads);
      mbar_init(bar(L::kSSmem + b), kGroupThreads);
      mbar_init(bar(L::kDReady + b), 1);
      mbar_init(bar(L::kDFree + b), kGroupThreads);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }

  // The schedule comes from a copy that completed before the first kernel of
  // the pass began, and Q, K, V from before that: every role but the one that
  // reads the start states runs ahead of the previous kernel's completion.
  const int i_begin = cta_begin[blockIdx.x];
  const int n = cta_begin[blockIdx.x + 1] - i_begin;
  const WorkTile* list = work + i_begin;
  int2* coord = reinterpret_cast<int2*>(smem + L::kCoord);
  // The producer's tile coordinates: loads issued before the CTA-wide set-up
  // completes, so their latency overlaps it.
  int2 c_lo = make_int2(0, 0), c_hi = make_int2(0, 0);
  if (warp == 0) {
    if (lane < n) c_lo = make_int2(list[lane].row0, list[lane].head);
    if (lane + 32 < n && lane + 32 < kCoordSlots) c_hi = make_int2(list[lane + 32].row0, list[lane + 32].head);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane < n) coord[lane] = c_lo;
    if (lane + 32 < n && lane + 32 < kCoordSlots) coord[lane + 32] = c_hi;
    __syncwarp();
    if (lane == 0) {
      bool ok = true;
      int i = 0;
      for (; i < n; ++i) {
        const int2 rc = i < kCoordSlots ? coord[i] : make_int2(list[i].row0, list[i].head);
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!wait_or_flag(bar(L::kEmpty + s), ph ^ 1, err, kErrTimeoutMma)) { ok = false; break; }
        const uint32_t st = base + L::kStage0 + s * kStageBytes;
        mbar_arrive_expect_tx(bar(L::kFull + s), kStageBytes);
        tma_load_3d(st + L::kQ, &tm_q, bar(L::kFull + s), 0, rc.x, rc.y);
        tma_load_3d(st + L::kK, &tm_k, bar(L::kFull + s), 0, rc.x, rc.y);
        tma_load_3d(st + L::kV, &tm_v, bar(L::kFull + s), 0, rc.x, rc.y);
      }
      // Wait (bounded) for the last loads to land before the CTA can exit.
      for (int u = (i > kStages ? i - kStages : 0); u < i; ++u)
        mbar_wait_bounded(bar(L::kFull + u % kStages), (u / kStages) & 1, ok ? kWaitLimitNs : 1000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ front issuer
    constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, 0, 0);
    constexpr uint32_t id_kv = idesc_bf16_f32(128, 64, 1, 1);
    WorkTile nxt = n > 0 ? load_tile(list) : WorkTile{};
    for (int i = 0; i < n; ++i) {
      const WorkTile r = nxt;
      if (i + 1 < n) nxt = load_tile(list + i + 1);
      const int s = i % kStages, b = i & 1;
      if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kFull + s), (i / kStages) & 1, err, kErrTimeoutTma)))
        break;
      const uint32_t st = base + L::kStage0 + s * kStageBytes;
      if (r.nrows < kTileRows) {
        // K and V rows past the tile may hold anything, even NaN; zero them so
        // masked P entries multiply zeros.  (A partial tile is the last of its
        // piece, so no state update reads them.)
        uint8_t* vrow = smem + (st + L::kV - base);
        uint8_t* krow = smem + (st + L::kK - base);
        for (int q = r.nrows * 8 + lane; q < kTileRows * 8; q += 32) {
          *reinterpret_cast<uint4*>(vrow + q * 16) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(krow + q * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      // P buffer b is free once P V of tile i-2 (which read it) has completed.
      bool ok = true;
      if (i >= 2) ok = wait_or_flag(bar(L::kOReady + b), ((i - 2) >> 1) & 1, err, kErrTimeoutMma);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after_sync();
      if (lane == 0) {
        const uint32_t colP = b ? kColP1 : kColP0;
        for (int kk = 0; kk < kHeadDim / 16; ++kk)
          mma_bf16(tmem + colP, smem_desc_sw128(st + L::kQ + kk * 32, 16, 1024),
                   smem_desc_sw128(st + L::kK + kk * 32, 16, 1024), id_qk, kk > 0);
        mma_commit(bar(L::kPReady + b));
      }
      __syncwarp();
      // dS region b is free once the state warps have read dS(i-2).
      if (i >= 2) ok = wait_or_flag(bar(L::kDFree + b), ((i - 2) >> 1) & 1, err, kErrTimeoutMma);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after_sync();
      if (lane == 0) {
        if (!(r.flags & kTileLast)) {
          // A = [K | K]^T (both 64-wide M atoms read the K tile: leading byte
          // offset 0), so TMEM lanes 64..127 hold a second copy of rows 0..63.
          const uint32_t colD = b ? kColD1 : kColD0;
          for (int kk = 0; kk < kTileRows / 16; ++kk)
            mma_bf16(tmem + colD, smem_desc_sw128(st + L::kK + kk * 2048, 0, 1024),
                     smem_desc_sw128(st + L::kV + kk * 2048, kRowTileBytes, 1024), id_kv, kk > 0);
        }
        mma_commit(bar(L::kDReady + b));
        mma_commit(bar(L::kEmpty + s));
      }
      __syncwarp();
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ O issuer
    constexpr uint32_t id_n64_b_mn = idesc_bf16_f32(128, 64, 0, 1);
    WorkTile nxt = n > 0 ? load_tile(list) : WorkTile{};
    for (int i = 0; i < n; ++i) {
      const WorkTile r = nxt;
      if (i + 1 < n) nxt = load_tile(list + i + 1);
      const int s = i % kStages, b = i & 1;
      const uint32_t st = base + L::kStage0 + s * kStageBytes;
      const bool has_state = !(r.flags & kTileFirst) || (r.flags & kTileHasInit);
      const uint32_t colO = b ? kColO1 : kColO0;
      // P(i) is bf16 in TMEM and the O buffer is free: O(i) = P(i) V(i).
      bool ok = wait_or_flag(bar(L::kPDone + b), (i >> 1) & 1, err, kErrTimeoutMma);
      if (ok && i >= 2) ok = wait_or_flag(bar(L::kOFree + b), ((i - 2) >> 1) & 1, err, kErrTimeoutMma);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after_sync();
      if (lane == 0) {
        const uint32_t colP = b ? kColP1 : kColP0;
        // keys 0..63 of P in columns 0..31, keys 64..127 in columns 64..95
        for (int kk = 0; kk < kTileRows / 16; ++kk)
          mma_bf16_tmem_a(tmem + colO, tmem + colP + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
                          smem_desc_sw128(st + L::kV + kk * 2048, kRowTileBytes, 1024),
                          id_n64_b_mn, kk > 0 ? 1u : 0u);
      }
      __syncwarp();
      // S(i) staged: O(i) += Q S_hi + Q S_lo; release the stage.
      if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kSSmem + b), (i >> 1) & 1, err, kErrTimeoutMma)))
        break;
      tc_fence_after_sync();
      if (lane == 0) {
        if (has_state) {
          const uint32_t sop = base + L::kS + b * kSOpBytes;
          for (int kk = 0; kk < kHeadDim / 16; ++kk)
            for (int part = 0; part < 2; ++part)
              mma_bf16(tmem + colO, smem_desc_sw128(st + L::kQ + kk * 32, 16, 1024),
                       smem_desc_sw128(sop + part * kStateTileBytes + kk * 2048, kStateTileBytes, 1024),
                       id_n64_b_mn, 1u);
        }
        mma_commit(bar(L::kOReady + b));
        mma_commit(bar(L::kEmpty + s));
      }
      __syncwarp();
    }
  } else if (warp < 3 + kConvWarps) {
    // ------------------------------------------------------------ P conversion
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    const int half = (warp - 3) >> 2;             // 64-column half of P this warp converts
    const int row = quarter * 32 + lane;          // tile row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    WorkTile nxt = n > 0 ? load_tile(list) : WorkTile{};
    for (int i = 0; i < n; ++i) {
      const WorkTile r = nxt;
      if (i + 1 < n) nxt = load_tile(list + i + 1);
      const int b = i & 1;
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
      const int hi_col = row < r.nrows ? row : -1;   // last kept column of this row
      const int c0 = half * 64, c1 = half * 64 + 63;
      // Warp-uniform shortcuts: this half-row block entirely kept or entirely masked.
      const bool all_kept = __all_sync(0xffffffffu, seg_start <= c0 && c1 <= hi_col);
      const bool all_zero = __all_sync(0xffffffffu, c0 > hi_col || c1 < seg_start);
      if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kPReady + b), (i >> 1) & 1, err, kErrTimeoutMma)))
        break;
      tc_fence_after_sync();
      const uint32_t colP = (b ? kColP1 : kColP0) + c0;
      uint32_t pk[32];
      if (all_zero) {
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = 0u;
      } else {
        uint32_t r0[32], r1[32];
        tmem_ld_32cols(tmem + lane_base + colP, r0);
        tmem_ld_32cols(tmem + lane_base + colP + 32, r1);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int jj = c0 + 2 * c;
          float p0 = __uint_as_float(c < 16 ? r0[2 * c] : r1[2 * c - 32]);
          float p1 = __uint_as_float(c < 16 ? r0[2 * c + 1] : r1[2 * c - 31]);
          if (!all_kept) {
            p0 = (jj >= seg_start && jj <= hi_col) ? p0 : 0.f;
            p1 = (jj + 1 >= seg_start && jj + 1 <= hi_col) ? p1 : 0.f;
          }
          pk[c] = pack_bf16x2(p0, p1);
        }
      }
      // bf16 pairs of this half's 64 columns go to its first 32 columns, all
      // of them read before any is overwritten.
      tmem_st_32cols(tmem + lane_base + colP, pk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kPDone + b));
    }
  } else {
    // ------------------------------------------------------------ state and output
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;          // tile row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    // State work: lanes 0..63 and their copy in lanes 64..127 hold state rows
    // d = row & 63; the lower copy handles columns 0..31, the upper 32..63.
    const int d = row & 63, sh = row >> 6;
    // The running state (row d, columns 32*sh ..) in fp32, and the first
    // term of the next piece's start state as loaded a tile ahead (summed
    // only when it is needed, so the loads stay in flight meanwhile).
    float s_run[32], s_a[32];
    // Which start state s_a holds, and which state each S operand holds
    // (first tile of a piece only; -1 = none / a running state).  A run of
    // pieces with the same start state (the packed branch tiles of one
    // parent) fetches and stages it once per operand.
    int64_t tag_a = -1, tag_op0 = -1, tag_op1 = -1;
    auto start_tag = [&](const WorkTile& r) -> int64_t {
      if (!(r.flags & kTileFirst) || !(r.flags & kTileHasInit)) return -1;
      return ((static_cast<int64_t>(r.stateA) + 1) << 40) ^ ((static_cast<int64_t>(r.stateB) + 1) << 16) ^
             static_cast<int64_t>(r.head);
    };

    // Issue the loads of the start state of the piece starting at tile record
    // `r`: the parent view's final state, or else the prefix slot.
    auto fetch_state = [&](const WorkTile& r) {
      const int64_t tag = start_tag(r);
      if (tag >= 0 && tag == tag_a) return;   // already in s_a
      tag_a = tag;
      const float4* a = nullptr;
      if (r.stateA >= 0)
        a = reinterpret_cast<const float4*>(
                stateA + ((static_cast<int64_t>(r.stateA) * H + r.head) * kHeadDim + d) * kHeadDim) + sh * 8;
      else if (r.stateB >= 0)
        a = reinterpret_cast<const float4*>(stateB + (static_cast<int64_t>(r.stateB) * kHeadDim + d) * kHeadDim) +
            sh * 8;
      if (a != nullptr) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 v4 = __ldcg(a + c);
          s_a[4 * c] = v4.x; s_a[4 * c + 1] = v4.y; s_a[4 * c + 2] = v4.z; s_a[4 * c + 3] = v4.w;
        }
      }
    };

    // The running state becomes the start state of the piece starting at `r`
    // (a piece with both terms -- a later piece of a long branch -- adds its
    // prefix slot here).
    auto start_piece = [&](const WorkTile& r) {
      const bool has = r.stateA >= 0 || r.stateB >= 0;
#pragma unroll
      for (int e = 0; e < 32; ++e) s_run[e] = has ? s_a[e] : 0.f;
      if (r.stateA >= 0 && r.stateB >= 0) {
        const float4* bb = reinterpret_cast<const float4*>(
            stateB + (static_cast<int64_t>(r.stateB) * kHeadDim + d) * kHeadDim) + sh * 8;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 v4 = __ldcg(bb + c);
          s_run[4 * c] += v4.x; s_run[4 * c + 1] += v4.y; s_run[4 * c + 2] += v4.z; s_run[4 * c + 3] += v4.w;
        }
      }
    };

    // S(t) -> S operand t & 1 (when tile t uses a state and the operand does
    // not hold that start state already).  The operand was last read by Q S
    // of tile t-2, whose completion o_work(t-2) saw.
    auto stage = [&](int t, const WorkTile& r) {
      const int64_t tag = start_tag(r);
      const bool uses = !(r.flags & kTileFirst) || (r.flags & kTileHasInit);
      const int64_t held = (t & 1) ? tag_op1 : tag_op0;
      if (uses && !(tag >= 0 && tag == held)) {
        stage_state_half_row(smem + L::kS + (t & 1) * kSOpBytes, d, sh, s_run);
        if (t & 1) tag_op1 = tag; else tag_op0 = tag;
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(L::kSSmem + (t & 1)));
    };

    // O(i) -> global (rows of the tile only).
    auto o_work = [&](int i, const WorkTile& r) -> bool {
      const int b = i & 1;
      if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kOReady + b), (i >> 1) & 1, err, kErrTimeoutMma)))
        return false;
      tc_fence_after_sync();
      const uint32_t colO = b ? kColO1 : kColO0;
      uint4* dst = reinterpret_cast<uint4*>(
          out + ((static_cast<int64_t>(r.row0) + row) * H + r.head) * kHeadDim);
      const bool store = row < r.nrows;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t r0[32];
        tmem_ld_32cols(tmem + lane_base + colO + 32 * h, r0);
        tmem_ld_wait();
        if (h == 1) {
          tc_fence_before_sync();
          mbar_arrive(bar(L::kOFree + b));
        }
        if (store) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            dst[4 * h + c] = make_uint4(pack_bf16x2(__uint_as_float(r0[8 * c]), __uint_as_float(r0[8 * c + 1])),
                                        pack_bf16x2(__uint_as_float(r0[8 * c + 2]), __uint_as_float(r0[8 * c + 3])),
                                        pack_bf16x2(__uint_as_float(r0[8 * c + 4]), __uint_as_float(r0[8 * c + 5])),
                                        pack_bf16x2(__uint_as_float(r0[8 * c + 6]), __uint_as_float(r0[8 * c + 7])));
        }
      }
      return true;
    };

    griddep_wait();   // start states from the scan
    if (n > 0) {
      WorkTile cur = load_tile(list);
      WorkTile nxt = n > 1 ? load_tile(list + 1) : WorkTile{};
      fetch_state(cur);
      start_piece(cur);
      stage(0, cur);
      if (n > 1 && (nxt.flags & kTileFirst)) fetch_state(nxt);
      bool ok = true;
      for (int i = 0; i < n && ok; ++i) {
        WorkTile nxt2 = i + 2 < n ? load_tile(list + i + 2) : WorkTile{};
        // S(i+1) first: the O issuer needs it right after P V of tile i+1.
        if (i + 1 < n) {
          const int b = i & 1;
          ok = __all_sync(0xffffffffu, wait_or_flag(bar(L::kDReady + b), (i >> 1) & 1, err, kErrTimeoutMma));
          if (!ok) break;
          tc_fence_after_sync();
          if (!(cur.flags & kTileLast)) {
            uint32_t r0[32];
            tmem_ld_32cols(tmem + lane_base + (b ? kColD1 : kColD0) + 32 * sh, r0);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) s_run[e] += __uint_as_float(r0[e]);
          } else {
            start_piece(nxt);
          }
          tc_fence_before_sync();
          mbar_arrive(bar(L::kDFree + b));
          stage(i + 1, nxt);
          // s_a is free again: fetch the start state of tile i+2 if it
          // begins a piece.
          if (i + 2 < n && (nxt2.flags & kTileFirst)) fetch_state(nxt2);
        }
        ok = o_work(i, cur);
        cur = nxt;
        nxt = nxt2;
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
  static std::atomic<uint64_t> done{0};
  cudaError_t e = set_smem_limit_once(span_output_kernel, bytes, done);
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
