// Tile-output kernel: the chunk output of view rows and the branch fork, in
// one launch (the third of the three launches of a pass).
//
// "Serving 0.88M TPS from Two RTXs and Mac Minis", section "Kernels" (each
// chunk: masked Q K^T times V inside the chunk plus Q times the state entering
// it; shared branch passes with the small kernels fused) and section "The
// Workload" (branches attend to the view but not to each other).
//
// A tile is up to 128 contiguous rows of one head: rows of one view, rows of
// one long branch, or several whole short branches with the same parent.  For
// row i of the tile, with start(i) the first row of i's segment inside the
// tile and S0 the tile's start state,
//
//     o_i = sum_{start(i) <= j <= i} (q_i . k_j) v_j  +  S0^T q_i .
//
// S0 is the exclusive chunk prefix from the scan (view tiles), the parent
// view's final state (branch tiles: the fork), or their sum (later tiles of a
// long branch).  A 128-row tile spans two 64-row chunks; the intra-tile mask
// covers the cross-chunk block exactly, so only the prefix of the tile's
// first chunk is read.
//
// Per CTA (128 threads, one tile row per thread = one TMEM lane):
//   TMA      Q, K, V tiles [128 rows][64] bf16, 128-byte swizzle
//   threads  S0 (fp32) -> bf16 high/low parts, MN-major B operand in smem
//   MMA      P = Q K^T            (M 128, N 128, K 64)   -> TMEM cols   0..127
//            O = Q S0_hi + Q S0_lo (M 128, N 64, K 64)   -> TMEM cols 128..191
//   threads  P row i: mask, -> bf16, K-major A operand in smem
//   MMA      O += P V             (M 128, N 64, K 128)
//   threads  O row i -> out (rows < nrows only)
// fp32 inputs arrive as bf16 high/low parts; every product then uses three
// MMAs (hi*hi + hi*lo + lo*hi) and P is split the same way.
#include "spanla_internal.h"
#include "tc_ptx.cuh"

namespace spanla {
namespace {

constexpr int kThreads = 128;
constexpr uint32_t kRowTileBytes = kTileRows * 128;         // 128 rows x 128 B = 16 KiB
constexpr uint32_t kStateTileBytes = kHeadDim * 128;        // 64 rows x 128 B = 8 KiB
constexpr uint32_t kPTileBytes = 2 * kRowTileBytes;         // 128 x 128 bf16 = 32 KiB
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemP = 0;
constexpr uint32_t kTmemO = 128;

template <int SPLIT>
struct TileSmem {
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + SPLIT * kRowTileBytes;
  static constexpr uint32_t kV = kK + SPLIT * kRowTileBytes;
  static constexpr uint32_t kS = kV + SPLIT * kRowTileBytes;     // S hi, S lo
  static constexpr uint32_t kP = kS + 2 * kStateTileBytes;       // P hi (, P lo)
  static constexpr uint32_t kBar = kP + SPLIT * kPTileBytes;
  static constexpr uint32_t kTmemSlot = kBar + 16;
  static constexpr uint32_t kBounds = kTmemSlot + 16;           // 128 x int32
  static constexpr uint32_t kBytes = kBounds + kTileRows * 4;
  static constexpr uint32_t kRequest = kBytes + 1024;
};

template <int SPLIT>
__global__ void __launch_bounds__(kThreads)
tile_output_kernel(const __grid_constant__ CUtensorMap tm_q0, const __grid_constant__ CUtensorMap tm_q1,
                   const __grid_constant__ CUtensorMap tm_k0, const __grid_constant__ CUtensorMap tm_k1,
                   const __grid_constant__ CUtensorMap tm_v0, const __grid_constant__ CUtensorMap tm_v1,
                   const TileDesc* __restrict__ tiles, const uint8_t* __restrict__ bounds,
                   const float* __restrict__ stateA, const float* __restrict__ stateB,
                   void* __restrict__ out, int H, unsigned* __restrict__ err) {
  using L = TileSmem<SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int h = blockIdx.y;
  const TileDesc td = tiles[blockIdx.x];

  const uint32_t bar_tma = base + L::kBar;
  const uint32_t bar_mma = base + L::kBar + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  int* sbounds = reinterpret_cast<int*>(smem + L::kBounds);

  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (tid < td.nbound) sbounds[tid] = bounds[td.bound0 + tid];
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();   // prefix states from the scan (and, through it, the bf16 parts)

  if (tid == 0) {
    mbar_arrive_expect_tx(bar_tma, 3 * SPLIT * kRowTileBytes);
    tma_load_3d(base + L::kQ, &tm_q0, bar_tma, 0, td.row0, h);
    tma_load_3d(base + L::kK, &tm_k0, bar_tma, 0, td.row0, h);
    tma_load_3d(base + L::kV, &tm_v0, bar_tma, 0, td.row0, h);
    if (SPLIT == 2) {
      tma_load_3d(base + L::kQ + kRowTileBytes, &tm_q1, bar_tma, 0, td.row0, h);
      tma_load_3d(base + L::kK + kRowTileBytes, &tm_k1, bar_tma, 0, td.row0, h);
      tma_load_3d(base + L::kV + kRowTileBytes, &tm_v1, bar_tma, 0, td.row0, h);
    }
  }

  // Start of this thread's row's segment inside the tile.
  const int i = tid;
  int seg_start = 0;
  for (int b = 0; b < td.nbound; ++b) {
    const int s = sbounds[b];
    if (s <= i) seg_start = s;
  }

  // Start state S0 = stateA[a] + stateB[b] -> bf16 high / low parts, stored
  // MN-major ([d rows][64 e], 128-byte swizzle) as the B operand of Q S0.
  const bool has_state = (td.stateA >= 0) || (td.stateB >= 0);
  if (has_state) {
    const int d = tid >> 1;
    const int e0 = (tid & 1) * 32;
    float s[32];
    const int64_t row_off = static_cast<int64_t>(h) * kStateFloats + d * kHeadDim + e0;
#pragma unroll
    for (int c = 0; c < 32; ++c) s[c] = 0.f;
    if (td.stateA >= 0) {
      const float4* a = reinterpret_cast<const float4*>(
          stateA + static_cast<int64_t>(td.stateA) * H * kStateFloats + row_off);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 x = a[c];
        s[4 * c] += x.x; s[4 * c + 1] += x.y; s[4 * c + 2] += x.z; s[4 * c + 3] += x.w;
      }
    }
    if (td.stateB >= 0) {
      const float4* b = reinterpret_cast<const float4*>(
          stateB + static_cast<int64_t>(td.stateB) * H * kStateFloats + row_off);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 x = b[c];
        s[4 * c] += x.x; s[4 * c + 1] += x.y; s[4 * c + 2] += x.z; s[4 * c + 3] += x.w;
      }
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float h0, l0, h1, l1;
        split_bf16(s[8 * g + 2 * u], h0, l0);
        split_bf16(s[8 * g + 2 * u + 1], h1, l1);
        hi[u] = pack_bf16x2(h0, h1);
        lo[u] = pack_bf16x2(l0, l1);
      }
      const uint32_t off = sw128_offset(d, e0 + 8 * g);
      *reinterpret_cast<uint4*>(smem + L::kS + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(smem + L::kS + kStateTileBytes + off) =
          make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }

  bool ok = mbar_wait_bounded(bar_tma, 0, kWaitLimitNs);
  if (!ok) {
    atomicOr(err, kErrTimeoutTma);
    mbar_wait_bounded(bar_tma, 0, kWaitLimitNs);
  }
  ok = __syncthreads_and(ok);

  if (ok) {
    // V rows past the tile's valid rows may hold anything (even NaN); zero
    // them so the masked P entries multiply zeros.
    if (i >= td.nrows) {
#pragma unroll
      for (int part = 0; part < SPLIT; ++part) {
        uint4* row = reinterpret_cast<uint4*>(smem + L::kV + part * kRowTileBytes + i * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) row[c] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();

  constexpr int kCombos = SPLIT == 2 ? 3 : 1;
  if (ok && tid == 0) {
    tc_fence_after_sync();
    // P = Q K^T
    constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, 0, 0);
    int n = 0;
    for (int kk = 0; kk < kHeadDim / 16; ++kk) {
      for (int combo = 0; combo < kCombos; ++combo) {
        const int pa = combo == 2 ? 1 : 0, pb = combo == 1 ? 1 : 0;
        const uint64_t a = smem_desc_sw128(base + L::kQ + pa * kRowTileBytes + kk * 32, 16, 1024);
        const uint64_t b = smem_desc_sw128(base + L::kK + pb * kRowTileBytes + kk * 32, 16, 1024);
        mma_bf16(tmem + kTmemP, a, b, id_qk, n++ > 0);
      }
    }
    // O = Q S0 (S0 split in high and low parts)
    if (has_state) {
      constexpr uint32_t id_qs = idesc_bf16_f32(128, 64, 0, 1);
      n = 0;
      for (int kk = 0; kk < kHeadDim / 16; ++kk) {
        for (int combo = 0; combo < (SPLIT == 2 ? 3 : 2); ++combo) {
          // bf16: Q*S_hi, Q*S_lo.  fp32: Q_hi*S_hi, Q_hi*S_lo, Q_lo*S_hi.
          const int pq = (SPLIT == 2 && combo == 2) ? 1 : 0;
          const int ps = combo == 1 ? 1 : 0;
          const uint64_t a = smem_desc_sw128(base + L::kQ + pq * kRowTileBytes + kk * 32, 16, 1024);
          const uint64_t b =
              smem_desc_sw128(base + L::kS + ps * kStateTileBytes + kk * 2048, kStateTileBytes, 1024);
          mma_bf16(tmem + kTmemO, a, b, id_qs, n++ > 0);
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
    // P row i -> mask -> bf16 (high, low) -> K-major A operand [128][128].
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {   // 32 columns at a time
      uint32_t r[32];
      tmem_ld_32cols(tmem + lane_base + kTmemP + cb * 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int g = 0; g < 4; ++g) {     // 8 columns = one 16-byte chunk
        const int j0 = cb * 32 + g * 8;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + 2 * u;
          float p0 = __uint_as_float(r[g * 8 + 2 * u]);
          float p1 = __uint_as_float(r[g * 8 + 2 * u + 1]);
          p0 = (j >= seg_start && j <= i && i < td.nrows) ? p0 : 0.f;
          p1 = (j + 1 >= seg_start && j + 1 <= i && i < td.nrows) ? p1 : 0.f;
          if (SPLIT == 2) {
            float h0, l0, h1, l1;
            split_bf16(p0, h0, l0);
            split_bf16(p1, h1, l1);
            hi[u] = pack_bf16x2(h0, h1);
            lo[u] = pack_bf16x2(l0, l1);
          } else {
            hi[u] = pack_bf16x2(p0, p1);
          }
        }
        const int blk = j0 >> 6;
        const uint32_t off = blk * kRowTileBytes + sw128_offset(i, j0 & 63);
        *reinterpret_cast<uint4*>(smem + L::kP + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if (SPLIT == 2)
          *reinterpret_cast<uint4*>(smem + L::kP + kPTileBytes + off) =
              make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();

  if (ok && tid == 0) {
    tc_fence_after_sync();
    // O += P V
    constexpr uint32_t id_pv = idesc_bf16_f32(128, 64, 0, 1);
    int n = has_state ? 1 : 0;
    for (int kk = 0; kk < kTileRows / 16; ++kk) {
      for (int combo = 0; combo < kCombos; ++combo) {
        const int pp = combo == 2 ? 1 : 0, pv = combo == 1 ? 1 : 0;
        const uint64_t a = smem_desc_sw128(
            base + L::kP + pp * kPTileBytes + (kk >> 2) * kRowTileBytes + (kk & 3) * 32, 16, 1024);
        const uint64_t b =
            smem_desc_sw128(base + L::kV + pv * kRowTileBytes + kk * 2048, kRowTileBytes, 1024);
        mma_bf16(tmem + kTmemO, a, b, id_pv, n++ > 0);
      }
    }
    mma_commit(bar_mma);
  }

  if (ok) {
    bool done = mbar_wait_bounded(bar_mma, 1, kWaitLimitNs);
    if (!done) {
      atomicOr(err, kErrTimeoutMma);
      mbar_wait_bounded(bar_mma, 1, kWaitLimitNs);
    }
    tc_fence_after_sync();
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t r0[32], r1[32];
    tmem_ld_32cols(tmem + lane_base + kTmemO, r0);
    tmem_ld_32cols(tmem + lane_base + kTmemO + 32, r1);
    tmem_ld_wait();
    if (done && i < td.nrows) {
      const int64_t row = (static_cast<int64_t>(td.row0) + i) * H + h;
      if (SPLIT == 2) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + row * kHeadDim);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          dst[c] = make_float4(__uint_as_float(r0[4 * c]), __uint_as_float(r0[4 * c + 1]),
                               __uint_as_float(r0[4 * c + 2]), __uint_as_float(r0[4 * c + 3]));
#pragma unroll
        for (int c = 0; c < 8; ++c)
          dst[8 + c] = make_float4(__uint_as_float(r1[4 * c]), __uint_as_float(r1[4 * c + 1]),
                                   __uint_as_float(r1[4 * c + 2]), __uint_as_float(r1[4 * c + 3]));
      } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + row * kHeadDim);
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

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_tile_output(bool split, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                               const CUtensorMap* tm_v, const TileDesc* tiles, int n_tiles,
                               const uint8_t* bounds, const float* stateA, const float* stateB,
                               void* out, int H, unsigned* err, cudaStream_t stream, bool pdl) {
  if (n_tiles <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_tiles, H);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (split) {
    auto kern = tile_output_kernel<2>;
    cfg.dynamicSmemBytes = TileSmem<2>::kRequest;
    static std::atomic<uint64_t> done{0};
    cudaError_t e = set_smem_limit_once(kern, static_cast<uint32_t>(cfg.dynamicSmemBytes), done);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, kern, tm_q[0], tm_q[1], tm_k[0], tm_k[1], tm_v[0], tm_v[1], tiles, bounds,
                              stateA, stateB, static_cast<void*>(out), H, err);
  }
  auto kern = tile_output_kernel<1>;
  cfg.dynamicSmemBytes = TileSmem<1>::kRequest;
  static std::atomic<uint64_t> done{0};
  cudaError_t e = set_smem_limit_once(kern, static_cast<uint32_t>(cfg.dynamicSmemBytes), done);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, kern, tm_q[0], tm_q[0], tm_k[0], tm_k[0], tm_v[0], tm_v[0], tiles, bounds,
                            stateA, stateB, static_cast<void*>(out), H, err);
}

}  // namespace spanla
