// Softmax-attention kernel (bf16 inputs) over the packed rows of a pass: the
// hybrid model's few softmax layers, on the same views and branches as its
// linear layers.
//
// "Serving 0.88M TPS from Two RTXs and Mac Minis", section "The Workload"
// (a branch sees its view and not its siblings) and section "Long Requests"
// (the softmax layers' K/V of a view is what a branch reuses).  Per head and
// query row t,
//
//     o_t = sum_j softmax_j(scale * q_t . k_j) v_j ,   lse_t = log sum_j exp(scale * q_t . k_j)
//
// over the keys row t sees: its own view's rows up to t, or, for a branch
// row, all of the parent view's rows and its own branch's rows up to t.
//
// Work unit = one SaItem: up to 128 query rows of one head and the sequence
// of 128-key blocks they attend to (prefix blocks, then own blocks; only the
// last own block -- the tile itself -- is masked).  Prefix blocks are read
// through their own pair of tensor maps: the pass's K and V for branches of
// views in the same pass, or K and V kept from the pass that ran the views.  Per key block g, with a
// reference maximum m and a running sum l per row (online softmax):
//
//     S_g = Q K_g^T                 (tcgen05, M128 N128 K64, fp32 in TMEM)
//     P_g = exp(scale (S_g - m))    (bf16, written back over S_g in TMEM)
//     O  += P_g V_g                 (tcgen05 with A = P_g from TMEM, M128 N64 K128,
//                                    accumulated in TMEM over the item's blocks)
//
// m is raised only when a row's block maximum exceeds it by more than
// 8 / (scale log2 e) (a factor of 2^8 in P): then O and l are first scaled by
// exp(scale (m_old - m_new)).  Below that, P stays within [0, 2^8] and the
// result is the same; the rescale (and with it a wait for the previous
// product) is rare.  At the end of an item, o = O / l.
//
// Persistent CTAs (one per SM) walk a host-built list of items.  11 warps:
//   warp 0     producer: Q of each item, K and V of each key block, by TMA
//              (Q double-buffered per item, K/V in a four-stage ring).
//   warp 1     S issuer (one lane): S_g as soon as block g has landed and
//              its TMEM buffer is free.  S/P has three TMEM buffers (g mod 3),
//              so S runs up to two blocks ahead of the softmax.
//   warp 10    O issuer (one lane): O += P_g V_g as soon as P_g is ready, into
//              the O buffer of the item (two, by item parity); it zeroes the V
//              rows past a partial block's keys and hands the stage back to
//              the producer.
//   warps 2-9  softmax: two warps per TMEM lane quarter, one query row per
//              thread in each; the warp of role g & 1 takes key block g whole
//              (all 128 columns of its rows): mask, block maximum, the raise
//              decision -- which needs the previous block's reference maximum,
//              handed over by the other warp through shared memory and
//              published again at once -- then exponentials, row sum and P
//              as bf16 in place.  So consecutive blocks' exponentials run in
//              the two warps at the same time, and only the short maximum /
//              decision step is ordered between them.  Each warp keeps its
//              own partial row sum; at the end of an item the two combine
//              and each writes half of the output columns (and lse).
#include "spanla_internal.h"
#include "tc_ptx.cuh"

namespace spanla {
namespace {

constexpr int kThreads = 352;
constexpr int kSoftmaxThreads = 256;
constexpr int kStages = 4;
constexpr uint32_t kTileBytes = kTileRows * 128;             // 128 rows x 128 B (bf16 x 64)
constexpr uint32_t kStageBytes = 2 * kTileBytes;             // K, V
constexpr uint32_t kTmemCols = 512;
// TMEM columns: three S/P buffers (128 each), two O accumulators (64 each).
constexpr int kSBufs = 3;
constexpr uint32_t kColO0 = 384, kColO1 = 448;
__device__ __forceinline__ uint32_t col_s(int g) { return static_cast<uint32_t>(g % kSBufs) * 128u; }

struct SaSmem {
  static constexpr uint32_t kQ = 0;                              // two Q tiles
  static constexpr uint32_t kStage0 = 2 * kTileBytes;
  static constexpr uint32_t kBar = kStage0 + kStages * kStageBytes;
  static constexpr int kFull = 0, kEmpty = kStages, kQFull = 2 * kStages, kQFree = kQFull + 2,
                       kSReady = kQFull + 4, kPDone = kSReady + kSBufs, kPVDone = kPDone + kSBufs,
                       kOReady = kPVDone + kSBufs, kOFree = kOReady + 2, kPair = kOFree + 2,
                       kDec = kPair + 4, kNumBars = kDec + 8;
  static constexpr uint32_t kTmemSlot = kBar + 8 * kNumBars;
  // Reference maximum after block g, [g & 1][row]; each role's partial row
  // sum and the maximum it is relative to at the end of an item,
  // [item parity][role][row].
  static constexpr uint32_t kDecM = kTmemSlot + 16;
  static constexpr uint32_t kRedL = kDecM + 2 * 128 * 4;
  static constexpr uint32_t kRedM = kRedL + 2 * 2 * 128 * 4;
  static constexpr uint32_t kBytes = kRedM + 2 * 2 * 128 * 4;
  static constexpr uint32_t kRequest = kBytes + 1024;
};
static_assert(SaSmem::kRequest <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ bool wait_or_flag(uint32_t bar, uint32_t parity, unsigned* err,
                                             unsigned code) {
  if (mbar_wait_bounded(bar, parity, kWaitLimitNs)) return true;
  atomicOr(err, code);
  return false;
}

__device__ __forceinline__ SaItem load_item(const SaItem* p) {
  SaItem t;
  const uint4* src = reinterpret_cast<const uint4*>(p);
  uint4* dst = reinterpret_cast<uint4*>(&t);
  dst[0] = __ldg(src);
  dst[1] = __ldg(src + 1);
  return t;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Paired fp32 arithmetic (one instruction for two lanes of a 64-bit register
// pair) and the three-input maximum, which halve the per-element instruction
// count of the softmax loops.
__device__ __forceinline__ uint64_t pair_f32(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpair_f32(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Key block jb of an item: first key row, valid keys, and whether it is the
// item's own (masked) diagonal block.
struct KeyBlock {
  int32_t kr0;
  int32_t cnt;
  bool diag;
};

__device__ __forceinline__ int32_t num_blocks(const SaItem& it) {
  return (it.pn + kTileRows - 1) / kTileRows + (it.r0 - it.os) / kTileRows + 1;
}

__device__ __forceinline__ KeyBlock key_block(const SaItem& it, int32_t jb) {
  const int32_t npre = (it.pn + kTileRows - 1) / kTileRows;
  if (jb < npre) return {it.ps + jb * kTileRows, min(kTileRows, it.pn - jb * kTileRows), false};
  const int32_t kr0 = it.os + (jb - npre) * kTileRows;
  return {kr0, kr0 == it.r0 ? it.nrows : kTileRows, kr0 == it.r0};
}

__global__ void __launch_bounds__(kThreads, 1)
softmax_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_pk,
                    const __grid_constant__ CUtensorMap tm_pv, const SaItem* __restrict__ items,
                    const int32_t* __restrict__ cta_begin, const uint8_t* __restrict__ bounds,
                    float scale_log2e, float scale, __nv_bfloat16* __restrict__ out,
                    float* __restrict__ lse, int H, unsigned* __restrict__ err) {
  using L = SaSmem;
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
      mbar_init(bar(L::kQFull + b), 1);
      mbar_init(bar(L::kQFree + b), 1);
      mbar_init(bar(L::kOReady + b), 1);
      mbar_init(bar(L::kOFree + b), kSoftmaxThreads);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(bar(L::kSReady + b), 1);
      mbar_init(bar(L::kPDone + b), kSoftmaxThreads / 2);   // the warps of the block's role
      mbar_init(bar(L::kPVDone + b), 1);
    }
    for (int q = 0; q < 4; ++q) {
      mbar_init(bar(L::kPair + q), 64);                       // the two warps of a lane quarter
      mbar_init(bar(L::kDec + 2 * q), 32);                    // decision of an even block
      mbar_init(bar(L::kDec + 2 * q + 1), 32);                // decision of an odd block
    }
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_pk);
    tma_prefetch_desc(&tm_pv);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const int i_begin = cta_begin[blockIdx.x];
  const int n = cta_begin[blockIdx.x + 1] - i_begin;
  const SaItem* list = items + i_begin;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      int g = 0;
      for (int i = 0; i < n && ok; ++i) {
        const SaItem it = load_item(list + i);
        const int qb = i & 1;
        if (!wait_or_flag(bar(L::kQFree + qb), ((i >> 1) & 1) ^ 1, err, kErrTimeoutMma)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(L::kQFull + qb), kTileBytes);
        tma_load_3d(base + L::kQ + qb * kTileBytes, &tm_q, bar(L::kQFull + qb), 0, it.r0, it.head);
        const int nb = num_blocks(it);
        for (int jb = 0; jb < nb; ++jb, ++g) {
          const KeyBlock kb = key_block(it, jb);
          const int s = g % kStages;
          if (!wait_or_flag(bar(L::kEmpty + s), ((g / kStages) & 1) ^ 1, err, kErrTimeoutMma)) { ok = false; break; }
          const uint32_t st = base + L::kStage0 + s * kStageBytes;
          mbar_arrive_expect_tx(bar(L::kFull + s), kStageBytes);
          // Prefix blocks come from the prefix arrays (the pass's own K and V,
          // or a parent view's K and V kept from an earlier pass).
          const bool pre = jb < (it.pn + kTileRows - 1) / kTileRows;
          tma_load_3d(st, pre ? &tm_pk : &tm_k, bar(L::kFull + s), 0, kb.kr0, it.head);
          tma_load_3d(st + kTileBytes, pre ? &tm_pv : &tm_v, bar(L::kFull + s), 0, kb.kr0, it.head);
        }
      }
      // Wait (bounded) for the loads in flight before the CTA can exit.
      for (int u = (g > kStages ? g - kStages : 0); u < g; ++u)
        mbar_wait_bounded(bar(L::kFull + u % kStages), (u / kStages) & 1, ok ? kWaitLimitNs : 1000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, 0, 0);
    int g = 0;
    bool ok = true;
    for (int i = 0; i < n && ok; ++i) {
      const SaItem it = load_item(list + i);
      const int qb = i & 1;
      const uint32_t qaddr = base + L::kQ + qb * kTileBytes;
      ok = __all_sync(0xffffffffu, wait_or_flag(bar(L::kQFull + qb), (i >> 1) & 1, err, kErrTimeoutTma));
      const int nb = num_blocks(it);
      for (int jb = 0; jb < nb && ok; ++jb, ++g) {
        const int s = g % kStages, sb = g % kSBufs;
        const uint32_t st = base + L::kStage0 + s * kStageBytes;
        bool w = wait_or_flag(bar(L::kFull + s), (g / kStages) & 1, err, kErrTimeoutTma);
        // S/P buffer sb was last read by P V of block g-3.
        if (w && g >= kSBufs) w = wait_or_flag(bar(L::kPVDone + sb), ((g - kSBufs) / kSBufs) & 1, err, kErrTimeoutMma);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after_sync();
        if (lane == 0) {
          const uint32_t colS = col_s(g);
          for (int kk = 0; kk < kHeadDim / 16; ++kk)
            mma_bf16(tmem + colS, smem_desc_sw128(qaddr + kk * 32, 16, 1024),
                     smem_desc_sw128(st + kk * 32, 16, 1024), id_qk, kk > 0 ? 1u : 0u);
          mma_commit(bar(L::kSReady + sb));
          if (jb == nb - 1) mma_commit(bar(L::kQFree + qb));
        }
        __syncwarp();
      }
    }
  } else if (warp == kThreads / 32 - 1) {
    // ------------------------------------------------------------ O issuer
    // O += P_g V_g once P_g is bf16 (and, at an item's first block, once the
    // softmax warps have read the O buffer's previous item); then the stage
    // (K read by S_g, which P_g depends on, and V) goes back to the producer.
    constexpr uint32_t id_pv = idesc_bf16_f32(128, 64, 0, 1);
    int g = 0;
    bool ok = true;
    for (int i = 0; i < n && ok; ++i) {
      const SaItem it = load_item(list + i);
      const int nb = num_blocks(it);
      const int ob = i & 1;
      const uint32_t colO = ob ? kColO1 : kColO0;
      for (int jb = 0; jb < nb && ok; ++jb, ++g) {
        const KeyBlock kb = key_block(it, jb);
        const int s = g % kStages, sb = g % kSBufs;
        const uint32_t st = base + L::kStage0 + s * kStageBytes;
        bool w = wait_or_flag(bar(L::kFull + s), (g / kStages) & 1, err, kErrTimeoutTma);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        if (kb.cnt < kTileRows) {
          // V rows past the block's keys may hold anything, even NaN (rows of
          // no segment); their P entries are 0, so make the rows 0 as well.
          uint8_t* vrow = smem + (st + kTileBytes - base);
          for (int q = kb.cnt * 8 + lane; q < kTileRows * 8; q += 32)
            *reinterpret_cast<uint4*>(vrow + q * 16) = make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
        }
        __syncwarp();
        w = wait_or_flag(bar(L::kPDone + sb), (g / kSBufs) & 1, err, kErrTimeoutMma);
        if (w && jb == 0 && i >= 2) w = wait_or_flag(bar(L::kOFree + ob), ((i - 2) >> 1) & 1, err, kErrTimeoutMma);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after_sync();
        if (lane == 0) {
          const uint32_t colS = col_s(g);
          // P of keys 0..63 is in columns 0..31 of the buffer, of keys
          // 64..127 in columns 64..95 (each written over its own scores).
          for (int kk = 0; kk < kTileRows / 16; ++kk)
            mma_bf16_tmem_a(tmem + colO, tmem + colS + kk * 8 + (kk >= 4 ? 32 : 0),
                            smem_desc_sw128(st + kTileBytes + kk * 2048, kTileBytes, 1024), id_pv,
                            (jb > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(L::kPVDone + sb));
          if (jb == nb - 1) mma_commit(bar(L::kOReady + ob));
          mma_commit(bar(L::kEmpty + s));
        }
        __syncwarp();
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    const int role = (warp - 2) >> 2;             // takes the key blocks g with g & 1 == role
    const int row = quarter * 32 + lane;          // query row in the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    float* dec_m = reinterpret_cast<float*>(smem + L::kDecM);
    float* red_l = reinterpret_cast<float*>(smem + L::kRedL);
    float* red_m = reinterpret_cast<float*>(smem + L::kRedM);
    // The two warps of a lane quarter meet at the end of an item (bounded
    // waits: a partner that gave up cannot hang this thread).
    const uint32_t pair_bar = bar(L::kPair + quarter);
    uint32_t pair_phase = 0;
    auto pair_sync = [&]() -> bool {
      mbar_arrive(pair_bar);
      const bool w = wait_or_flag(pair_bar, pair_phase & 1, err, kErrTimeoutMma);
      ++pair_phase;
      return __all_sync(0xffffffffu, w);
    };
    // Raise m only when a block maximum exceeds it by this much (raw score
    // units): P then stays below 2^8.
    const float raise_margin = 8.f / scale_log2e;
    // This warp's partial row sum over its blocks of the current item, and the
    // reference maximum it is relative to.
    float l_w = 0.f, m_w = -INFINITY;
    float l_done = 0.f, m_done = -INFINITY;
    SaItem done_it{};        // item whose output is still to be written
    int done_idx = -1;
    int g = 0;

    // Bring l_w to reference maximum m.
    auto rebase = [&](float m) {
      if (m != m_w) {
        l_w = m_w == -INFINITY ? 0.f : l_w * ex2((m_w - m) * scale_log2e);
        m_w = m;
      }
    };

    // O of item `it` (index ii) / l -> global row (this role's 32 output
    // columns); lse = scale * m + log(l).  l combines both roles' sums.
    auto finish = [&](const SaItem& it, int ii, float m_part, float l_part) -> bool {
      const int ob = ii & 1;
      red_l[(ob * 2 + role) * 128 + row] = l_part;
      red_m[(ob * 2 + role) * 128 + row] = m_part;
      if (!pair_sync()) return false;
      const float l_o = red_l[(ob * 2 + (role ^ 1)) * 128 + row];
      const float m_o = red_m[(ob * 2 + (role ^ 1)) * 128 + row];
      const float m = fmaxf(m_part, m_o);
      const float l = (m_part == -INFINITY ? 0.f : l_part * ex2((m_part - m) * scale_log2e)) +
                      (m_o == -INFINITY ? 0.f : l_o * ex2((m_o - m) * scale_log2e));
      if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kOReady + ob), (ii >> 1) & 1, err, kErrTimeoutMma)))
        return false;
      tc_fence_after_sync();
      uint32_t r0[32];
      tmem_ld_32cols(tmem + lane_base + (ob ? kColO1 : kColO0) + 32 * role, r0);
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kOFree + ob));
      if (row < it.nrows) {
        const float inv = 1.f / l;
        uint4* dst = reinterpret_cast<uint4*>(out + ((static_cast<int64_t>(it.r0) + row) * H + it.head) * kHeadDim) +
                     4 * role;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          dst[c] = make_uint4(pack_bf16x2(__uint_as_float(r0[8 * c]) * inv, __uint_as_float(r0[8 * c + 1]) * inv),
                              pack_bf16x2(__uint_as_float(r0[8 * c + 2]) * inv, __uint_as_float(r0[8 * c + 3]) * inv),
                              pack_bf16x2(__uint_as_float(r0[8 * c + 4]) * inv, __uint_as_float(r0[8 * c + 5]) * inv),
                              pack_bf16x2(__uint_as_float(r0[8 * c + 6]) * inv, __uint_as_float(r0[8 * c + 7]) * inv));
        if (lse != nullptr && role == 0) lse[(static_cast<int64_t>(it.r0) + row) * H + it.head] = scale * m + logf(l);
      }
      return true;
    };

    // 64 scores (key columns [c0, c0 + 64) of block g) with keys outside
    // [lo, hi] masked to -inf.
    auto load_half = [&](uint32_t colS, int c0, int lo, int hi, float (&x)[64]) {
      uint32_t sr[64];
      tmem_ld_32cols(tmem + lane_base + colS + c0, *reinterpret_cast<uint32_t(*)[32]>(sr));
      tmem_ld_32cols(tmem + lane_base + colS + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
      tmem_ld_wait();
      if (__all_sync(0xffffffffu, lo <= c0 && hi >= c0 + 63)) {
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(sr[c]);
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = (c0 + c >= lo && c0 + c <= hi) ? __uint_as_float(sr[c]) : -INFINITY;
      }
    };
    // P of 64 scores against reference maximum m, as bf16 into the first 32
    // of their columns; returns their sum.
    auto exp_store = [&](uint32_t colS, int c0, float m, const float (&x)[64]) -> float {
      const float neg = -(m == -INFINITY ? 0.f : m) * scale_log2e;
      const uint64_t c2 = pair_f32(scale_log2e, scale_log2e), n2 = pair_f32(neg, neg);
      uint64_t acc0 = pair_f32(0.f, 0.f), acc1 = acc0;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float x0, x1;
        unpair_f32(fma_f32x2(pair_f32(x[2 * c], x[2 * c + 1]), c2, n2), x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        if (c & 1) acc1 = add_f32x2(acc1, pair_f32(p0, p1));
        else acc0 = add_f32x2(acc0, pair_f32(p0, p1));
        pk[c] = pack_bf16x2(p0, p1);
      }
      tmem_st_32cols(tmem + lane_base + colS + c0, pk);
      float a0, a1, b0, b1;
      unpair_f32(acc0, a0, a1);
      unpair_f32(acc1, b0, b1);
      return (a0 + b0) + (a1 + b1);
    };

    bool ok = true;
    for (int i = 0; i < n && ok; ++i) {
      const SaItem it = load_item(list + i);
      const int ob = i & 1;
      int seg_start = 0;
      for (int q = 0; q < it.nseg; ++q) {
        const int sb = bounds[it.seg0 + q];
        if (sb <= row) seg_start = sb;
      }
      const int hi_col = row < it.nrows ? row : -1;   // last visible key of the diagonal block
      const int nb = num_blocks(it);
      for (int jb = 0; jb < nb && ok; ++jb, ++g) {
        if (jb == 0) {
          // A new item: this warp's partial sum starts again; the previous
          // item (whose last product lands soon) is written out.
          l_done = l_w;
          m_done = m_w;
          l_w = 0.f;
          m_w = -INFINITY;
          if (done_idx >= 0) {
            if (!finish(done_it, done_idx, m_done, l_done)) { ok = false; break; }
            done_idx = -1;
          }
        }
        if (jb == nb - 1) {
          done_it = it;
          done_idx = i;
        }
        if ((g & 1) != role) continue;
        const KeyBlock kb = key_block(it, jb);
        const int sb = g % kSBufs;
        // Visible key columns of the row: [lo, hi] (0..127).
        int lo = 0, hi = 127;
        if (kb.diag) {
          lo = seg_start;
          hi = hi_col;
        } else if (kb.cnt < kTileRows) {
          hi = kb.cnt - 1;
        }
        if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kSReady + sb), (g / kSBufs) & 1, err, kErrTimeoutMma))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t colS = col_s(g);
        float x[64];
        load_half(colS, 0, lo, hi, x);
        float mx0 = fmaxf(x[0], x[1]), mx1 = fmaxf(x[2], x[3]);
#pragma unroll
        for (int c = 4; c < 64; c += 4) {
          mx0 = max3(mx0, x[c], x[c + 1]);
          mx1 = max3(mx1, x[c + 2], x[c + 3]);
        }
        load_half(colS, 64, lo, hi, x);
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          mx0 = max3(mx0, x[c], x[c + 1]);
          mx1 = max3(mx1, x[c + 2], x[c + 3]);
        }
        const float mx = fmaxf(mx0, mx1);
        // The reference maximum after block g-1, handed over by the other
        // warp (every block hands one over, so the two stay in step).
        float m_ref = -INFINITY;
        if (g >= 1) {
          const int gp = g - 1;
          if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kDec + 2 * quarter + (gp & 1)), (gp >> 1) & 1, err,
                                                    kErrTimeoutMma))) {
            ok = false;
            break;
          }
          m_ref = dec_m[(gp & 1) * 128 + row];
        }
        if (jb == 0) {
          m_ref = mx;   // the item's O starts from this block (no rescale)
        } else if (__any_sync(0xffffffffu, mx > m_ref + raise_margin)) {
          // Raise m for the rows that need it: O (after the previous block's
          // product has landed) scales by exp(scale (m_old - m_new)); the
          // partial sums follow when they are next used.
          const int gp = g - 1, sp = gp % kSBufs;
          if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kPVDone + sp), (gp / kSBufs) & 1, err, kErrTimeoutMma))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const float m_new = fmaxf(m_ref, mx);
          const float alpha = m_new == m_ref ? 1.f : ex2((m_ref - m_new) * scale_log2e);   // 0 when m_ref = -inf
          const uint32_t colO = ob ? kColO1 : kColO0;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t r0[32];
            tmem_ld_32cols(tmem + lane_base + colO + 32 * h, r0);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) r0[c] = __float_as_uint(__uint_as_float(r0[c]) * alpha);
            tmem_st_32cols(tmem + lane_base + colO + 32 * h, r0);
          }
          m_ref = m_new;
        }
        // Hand the decision to the other warp before the exponentials.
        dec_m[(g & 1) * 128 + row] = m_ref;
        mbar_arrive(bar(L::kDec + 2 * quarter + (g & 1)));
        rebase(m_ref);
        // Keys 64..127 are in registers; keys 0..63 are read again.
        float sum = exp_store(colS, 64, m_ref, x);
        load_half(colS, 0, lo, hi, x);
        sum += exp_store(colS, 0, m_ref, x);
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(bar(L::kPDone + sb));
        l_w += sum;
      }
    }
    if (ok && done_idx >= 0) finish(done_it, done_idx, m_w, l_w);
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_softmax_attn(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                const CUtensorMap* tm_v, const CUtensorMap* tm_pk,
                                const CUtensorMap* tm_pv, const SaItem* items,
                                const int32_t* cta_begin, int grid, const uint8_t* bounds,
                                float scale_log2e, float scale, void* out, float* lse, int H,
                                unsigned* err, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  const uint32_t bytes = SaSmem::kRequest;
  static std::atomic<uint64_t> done{0};
  cudaError_t e = set_smem_limit_once(softmax_attn_kernel, bytes, done);
  if (e != cudaSuccess) return e;
  softmax_attn_kernel<<<grid, kThreads, bytes, stream>>>(tm_q[0], tm_k[0], tm_v[0], tm_pk[0], tm_pv[0], items,
                                                         cta_begin, bounds,
                                                         scale_log2e, scale,
                                                         static_cast<__nv_bfloat16*>(out), lse, H, err);
  return cudaGetLastError();
}

}  // namespace spanla
