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
//              thread pair, each thread of the pair on one half of the 128
//              key columns (and one half of the 64 output columns): mask,
//              block maximum (the pair swaps its halves' maxima through
//              shared memory), exponentials, row sum, P as bf16 in place; at
//              the end of an item O / l (and lse) to global memory.
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
                       kNumBars = kPair + 4;
  static constexpr uint32_t kTmemSlot = kBar + 8 * kNumBars;
  // Row maxima of the two column halves, [block parity][half][row], and row
  // sums at the end of an item, [item parity][half][row].
  static constexpr uint32_t kRedMax = kTmemSlot + 16;
  static constexpr uint32_t kRedSum = kRedMax + 2 * 2 * 128 * 4;
  static constexpr uint32_t kBytes = kRedSum + 2 * 2 * 128 * 4;
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
      mbar_init(bar(L::kPDone + b), kSoftmaxThreads);
      mbar_init(bar(L::kPVDone + b), 1);
    }
    for (int q = 0; q < 4; ++q) mbar_init(bar(L::kPair + q), 64);   // the two warps of a lane quarter
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
          // 64..127 in columns 64..95 (one column half per softmax thread).
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
    const int half = (warp - 2) >> 2;             // key columns [64 half, 64 half + 64)
    const int row = quarter * 32 + lane;          // query row in the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    float* red_max = reinterpret_cast<float*>(smem + L::kRedMax);
    float* red_sum = reinterpret_cast<float*>(smem + L::kRedSum);
    // The two threads of a row meet on their lane quarter's mbarrier, one
    // phase per exchange (bounded waits: a partner that gave up cannot hang
    // this thread).
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
    float m_ref = -INFINITY, l_run = 0.f;
    float m_done = 0.f, l_done = 1.f;
    SaItem done_it{};        // item whose output is still to be written
    int done_idx = -1;
    int g = 0;

    // O of item `it` (index ii) / l -> global row; lse = scale * m + log(l).
    // l is the sum of the pair's two partial sums.
    auto finish = [&](const SaItem& it, int ii, float m, float l_part) -> bool {
      const int ob = ii & 1;
      float* rs = red_sum + ob * 256;
      rs[half * 128 + row] = l_part;
      if (!pair_sync()) return false;
      const float l = l_part + rs[(half ^ 1) * 128 + row];
      if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kOReady + ob), (ii >> 1) & 1, err, kErrTimeoutMma)))
        return false;
      tc_fence_after_sync();
      uint32_t r0[32];
      tmem_ld_32cols(tmem + lane_base + (ob ? kColO1 : kColO0) + 32 * half, r0);
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kOFree + ob));
      if (row < it.nrows) {
        const float inv = 1.f / l;
        uint4* dst = reinterpret_cast<uint4*>(out + ((static_cast<int64_t>(it.r0) + row) * H + it.head) * kHeadDim) +
                     4 * half;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          dst[c] = make_uint4(pack_bf16x2(__uint_as_float(r0[8 * c]) * inv, __uint_as_float(r0[8 * c + 1]) * inv),
                              pack_bf16x2(__uint_as_float(r0[8 * c + 2]) * inv, __uint_as_float(r0[8 * c + 3]) * inv),
                              pack_bf16x2(__uint_as_float(r0[8 * c + 4]) * inv, __uint_as_float(r0[8 * c + 5]) * inv),
                              pack_bf16x2(__uint_as_float(r0[8 * c + 6]) * inv, __uint_as_float(r0[8 * c + 7]) * inv));
        if (lse != nullptr && half == 0) lse[(static_cast<int64_t>(it.r0) + row) * H + it.head] = scale * m + logf(l);
      }
      return true;
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
        const KeyBlock kb = key_block(it, jb);
        const int b = g & 1, sb = g % kSBufs;
        if (jb == 0) {
          m_done = m_ref;
          l_done = l_run;
          m_ref = -INFINITY;
          l_run = 0.f;
        }
        // Visible key columns of this thread's half: [lo, hi] (relative to 64 half).
        int lo = 0, hi = 63;
        if (kb.diag) {
          lo = seg_start - 64 * half;
          hi = hi_col - 64 * half;
        } else if (kb.cnt < kTileRows) {
          hi = kb.cnt - 1 - 64 * half;
        }
        if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kSReady + sb), (g / kSBufs) & 1, err, kErrTimeoutMma))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t colS = col_s(g) + 64 * half;
        uint32_t sr[64];
        tmem_ld_32cols(tmem + lane_base + colS, *reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_ld_32cols(tmem + lane_base + colS + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
        tmem_ld_wait();
        float s[64];
        if (__all_sync(0xffffffffu, lo <= 0 && hi >= 63)) {
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = (c >= lo && c <= hi) ? __uint_as_float(sr[c]) : -INFINITY;
        }
        float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
#pragma unroll
        for (int c = 4; c < 64; c += 4) {
          mx0 = max3(mx0, s[c], s[c + 1]);
          mx1 = max3(mx1, s[c + 2], s[c + 3]);
        }
        float* rm = red_max + b * 256;
        rm[half * 128 + row] = fmaxf(mx0, mx1);
        if (!pair_sync()) { ok = false; break; }
        const float mx = fmaxf(fmaxf(mx0, mx1), rm[(half ^ 1) * 128 + row]);
        if (jb == 0) {
          m_ref = mx;   // the item's O starts from this block (no rescale)
        } else if (__any_sync(0xffffffffu, mx > m_ref + raise_margin)) {
          // Raise m for the rows that need it: O (after the previous block's
          // product has landed) and l scale by exp(scale (m_old - m_new)).
          const int gp = g - 1, sp = gp % kSBufs;
          if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kPVDone + sp), (gp / kSBufs) & 1, err, kErrTimeoutMma))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const float m_new = fmaxf(m_ref, mx);
          const float alpha = m_new == m_ref ? 1.f : ex2((m_ref - m_new) * scale_log2e);   // 0 when m_ref = -inf
          const uint32_t colO = (ob ? kColO1 : kColO0) + 32 * half;
          uint32_t r0[32];
          tmem_ld_32cols(tmem + lane_base + colO, r0);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) r0[c] = __float_as_uint(__uint_as_float(r0[c]) * alpha);
          tmem_st_32cols(tmem + lane_base + colO, r0);
          l_run *= alpha;
          m_ref = m_new;
        }
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        const float neg = -m_use * scale_log2e;
        // p = 2^(s c - m c) two lanes at a time; two paired partial sums.
        const uint64_t c2 = pair_f32(scale_log2e, scale_log2e), n2 = pair_f32(neg, neg);
        uint64_t acc0 = pair_f32(0.f, 0.f), acc1 = acc0;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float x0, x1;
          unpair_f32(fma_f32x2(pair_f32(s[2 * c], s[2 * c + 1]), c2, n2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          if (c & 1) acc1 = add_f32x2(acc1, pair_f32(p0, p1));
          else acc0 = add_f32x2(acc0, pair_f32(p0, p1));
          pk[c] = pack_bf16x2(p0, p1);
        }
        float a0, a1, b0, b1;
        unpair_f32(acc0, a0, a1);
        unpair_f32(acc1, b0, b1);
        const float sum0 = a0 + b0, sum1 = a1 + b1;
        // The 64 bf16 of this half's P go over the first 32 of its columns.
        tmem_st_32cols(tmem + lane_base + colS, pk);
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(bar(L::kPDone + sb));
        l_run += sum0 + sum1;
        // The previous item is complete once its last product has landed:
        // write it out now that this item's first block is under way.
        if (jb == 0 && done_idx >= 0) {
          if (!finish(done_it, done_idx, m_done, l_done)) { ok = false; break; }
          done_idx = -1;
        }
        if (jb == nb - 1) {
          done_it = it;
          done_idx = i;
        }
      }
    }
    if (ok && done_idx >= 0) finish(done_it, done_idx, m_ref, l_run);
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
