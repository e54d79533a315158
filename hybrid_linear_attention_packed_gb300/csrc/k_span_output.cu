// Span-output kernel (bf16 inputs): the output of every view row and every
// branch row, carrying the state across the tiles of a piece -- and, as the
// one-launch pass, the piece states and the prefix sums as well.
//
// "Serving 0.88M TPS from Two RTXs and Mac Minis", section "Kernels" (each
// 64-token chunk: a masked Q K^T times V inside the chunk plus Q times the
// state entering it; one scan per pass; shared branch passes with the small
// kernels fused) and section "The Workload" (branches attend to the view, not
// to each other).
//
// Each CTA runs one contiguous run of (tile, head) work from a host-built
// list.  A piece is the part of one view-head or long-branch-head inside the
// run; a tile of packed short branches is a piece of its own.  With S the
// state entering a tile (the piece's start state for its first tile), every
// row i of the tile gets
//
//     o_i = sum_{start(i) <= j <= i} (q_i . k_j) v_j  +  S^T q_i ,
//
// and the next tile of the piece starts from S + K^T V of this one.
//
// Start states.  With three launches (span_state -> scan -> this kernel) a
// piece's start state is one scanned prefix slot plus, for branches, the
// parent view's final state written by the scan.  In the one-launch pass
// (fused) this kernel first sums K^T V over its own pieces whose state other
// CTAs need (phase 1, written to workspace slots), counts itself in a global
// counter, and a CTA whose pieces start from other CTAs' states waits until
// every phase-1 CTA has counted itself (the grid is launched cooperatively,
// so every CTA is resident) and sums those slots itself: no scan.  The CTA
// that holds the last tile of a view-head computes the view's final state
// on chip (K^T V of that tile added to the running state), writes it out and
// starts that view's following branch tiles in its run from it directly.
//
// Software pipelined over consecutive tiles t.  19 warps:
//   warp 0     producer: phase-1 K, V tiles, then Q, K, V tiles by TMA into
//              a four-stage ring.  When a pass's phase-1 K and V exceed what
//              the L2 can keep for the tiles' second read, the phase-1 loads
//              take the L2 evict-first policy (the kP1EvictFirst instance),
//              so that they displace one another rather than dirty lines
//              that would first have to be written back.
//   warp 1     front issuer (one lane; the warp zeroes partial-tile K/V
//              rows): phase 1, K^T V summed over each phase-1 piece into a
//              TMEM region; then per tile, as soon as it has landed,
//              P(t) = Q K^T  (M128 N128 K64) into TMEM buffer t & 1, then,
//              unless t ends its piece (or when it ends a view-head), the
//              tile's own state  dS(t) = K^T V  (M128 N64 K128) into TMEM
//              region t & 1.
//   warp 2     O issuer (one lane): once the P conversion has turned P(t)
//              into bf16 in place,  O(t) = P(t) V  (M128 N64 K128, P read
//              from tensor memory), which hands P buffer t & 1 back to the
//              front issuer as soon as it completes, then, with S(t) staged,
//              O(t) += Q S  (M128 N64 K64, S rounded to bf16), so that an O
//              buffer is held only from the end of the conversion until the
//              tile's output is read.
//   warps 3-10 P conversion, two warps per TMEM lane quarter, one per
//              64-column half: each thread owns one tile row (TMEM lane) and
//              turns its half of P(t) into the masked bf16 A operand in place
//              in tensor memory, 32 columns at a time -- 64 fp32 columns
//              become 64 bf16 in the half's first 32 columns (P V reads keys
//              0..63 from columns 0..31 and keys 64..127 from columns 64..95).
//   warps 11-18 state and output, two warps per lane quarter.  Phase 1: the
//              piece states out of TMEM into the workspace.  Then they hold
//              the running fp32 state in registers (16 columns of one state
//              row per thread); per step t they add dS(t) to it (or load the
//              next piece's start state), stage S(t+1) rounded to bf16 for
//              Q S, and then store O(t), 32 of its 64 columns per warp (one
//              32 x 32 TMA store when the warp's rows all lie in the tile).
// K^T V runs with M = 128 and the K tile as both 64-wide M atoms, so TMEM
// lanes 64..127 hold a copy of rows 0..63: the lower copy is read for
// columns 0..31, the upper for 32..63.
#include "spanla_internal.h"
#include "tc_ptx.cuh"

namespace spanla {
namespace {

constexpr int kThreads = 32 * (3 + 8 + 8);
constexpr int kGroupWarps = 8;                           // state and output
constexpr int kGroupThreads = 32 * kGroupWarps;
constexpr int kConvWarps = 8;                            // P conversion
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kStateWarp0 = 3 + kConvWarps;              // first state/output warp
constexpr int kStages = 4;
constexpr uint32_t kRowTileBytes = kTileRows * 128;        // 128 rows x 128 B
constexpr uint32_t kStageBytes = 3 * kRowTileBytes;       // Q K V
constexpr uint32_t kStateTileBytes = kHeadDim * 128;       // 64 rows x 128 B (bf16)
// An S operand: S in bf16 in its first 8 KB.  Its second 8 KB holds O of
// two lane quarters on its way out (quarters 0, 1 in operand 0; 2, 3 in
// operand 1), and the whole 16 KB also serves as the fp32 buffer of the
// start-state sums.
constexpr uint32_t kSOpBytes = 2 * kStateTileBytes;
constexpr uint32_t kOQuarterBytes = kOutStoreRows * 128;     // 32 rows of O (bf16) on their way out
static_assert(kOutStoreRows == 32, "one TMA store per warp's rows");
static_assert(kFirstLoads <= kStages, "the set-up loads use fresh stages");
static_assert(2 * kOQuarterBytes == kStateTileBytes, "two quarters of O staging per S operand");
constexpr int kCoordSlots = 64;                              // tile coordinates staged for the producer
constexpr int kP1Slots = 32;                                 // phase-1 piece records staged
constexpr uint32_t kTmemCols = 512;
// TMEM columns: P buffers (128 each), O buffers (64 each), dS regions (64 each).
constexpr uint32_t kColP0 = 0, kColP1 = 128, kColO0 = 256, kColO1 = 320, kColD0 = 384, kColD1 = 448;
constexpr uint32_t kNamedStateBar = 1;                       // bar.sync id of the state warps

struct OutSmem {
  static constexpr uint32_t kStage0 = 0;
  static constexpr uint32_t kQ = 0, kK = kRowTileBytes, kV = 2 * kRowTileBytes;
  static constexpr uint32_t kS = kStages * kStageBytes;          // two S operands (S, O staging)
  static constexpr uint32_t kBar = kS + 2 * kSOpBytes;
  // barrier slots (8 bytes each); the pairs are used by alternate tiles (or
  // phase-1 pieces).  Empty takes two arrivals per use: the front issuer's
  // and the O issuer's MMAs both read a tile's stage (the front issuer
  // arrives twice on a phase-1 stage).  PFree (P V done: the P buffer may be
  // overwritten) is apart from OReady (P V and Q S done), so that the next
  // Q K^T into a P buffer does not wait for the state staging Q S waits for.
  static constexpr int kFull = 0, kEmpty = kStages, kPReady = 2 * kStages,
                       kPDone = kPReady + 2, kOReady = kPReady + 4, kOFree = kPReady + 6,
                       kSSmem = kPReady + 8, kDReady = kPReady + 10, kDFree = kPReady + 12,
                       kP1Ready = kPReady + 14, kP1Free = kPReady + 16, kP1Done = kPReady + 18,
                       kPFree = kPReady + 19, kNumBars = kPReady + 21;
  static constexpr uint32_t kTmemSlot = kBar + 8 * kNumBars;
  static constexpr uint32_t kCoord = kTmemSlot + 8;              // (row0, head) of the first tiles
  static constexpr uint32_t kP1 = kCoord + 8 * kCoordSlots;      // phase-1 piece records
  static constexpr uint32_t kBytes = kP1 + sizeof(SpanDesc) * kP1Slots;
  static constexpr uint32_t kRequest = kBytes + 1024;
};
static_assert(OutSmem::kRequest <= 227 * 1024, "shared memory budget");

// Kernel parameters besides the tensor maps (see SpanOutputArgs).
struct OutParams {
  const CtaHead* heads;
  const WorkTile* work;
  const int32_t* cta_begin;
  const uint8_t* bounds;
  const float* stateA;
  float* ws;
  float* final_out;
  __nv_bfloat16* out;
  unsigned* err;
  const SpanDesc* p1;
  const int32_t* p1_begin;
  unsigned* counter;
  int a_rows;
  int H;
  int fused;
  int n_p1_ctas;
};

__device__ __forceinline__ bool wait_or_flag(uint32_t bar, uint32_t parity, unsigned* err,
                                             unsigned code) {
  if (mbar_wait_bounded(bar, parity, kWaitLimitNs)) return true;
  atomicOr(err, code);
  return false;
}

// The parts of a tile record each role reads (fewer registers per role).
struct TileHead {     // row0, nrows, head, flags
  int32_t row0, nrows, head, flags;
};
struct TileState {    // ... and the start-state recipe
  int32_t row0, nrows, head, flags, stateA, stateB, a_n, b_n, final_idx;
};
struct TileMask {     // rows and segment starts (P conversion)
  int32_t nrows, bound0, nbound;
  uint4 inl;
};

__device__ __forceinline__ TileHead load_head(const WorkTile* p) {
  const int4 a = __ldg(reinterpret_cast<const int4*>(p));
  return TileHead{a.x, a.y, a.z, a.w};
}

__device__ __forceinline__ TileState load_state(const WorkTile* p) {
  const int4 a = __ldg(reinterpret_cast<const int4*>(p));
  const int4 b = __ldg(reinterpret_cast<const int4*>(p) + 1);
  const int32_t f = __ldg(&p->final_idx);
  return TileState{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, f};
}

__device__ __forceinline__ TileMask load_mask(const WorkTile* p) {
  const int4 c = __ldg(reinterpret_cast<const int4*>(p) + 2);
  const uint4 d = __ldg(reinterpret_cast<const uint4*>(p) + 3);
  return TileMask{__ldg(&p->nrows), c.y, c.z, d};
}

__device__ __forceinline__ int inline_bound(const uint4& v, int q) {
  const uint32_t w = q < 4 ? v.x : q < 8 ? v.y : q < 12 ? v.z : v.w;
  return static_cast<int>((w >> (8 * (q & 3))) & 0xffu);
}

// Write 16 state values (columns col0 ..) of row d, rounded to bf16, into
// the MN-major S operand ([d][64 e], 128-byte swizzle).  (The state itself
// stays fp32; only its product with Q takes the rounded copy, whose entries
// are off by less than 2^-9 of their value, as q, k and v are.)
__device__ __forceinline__ void stage_state_slice(uint8_t* s_op, int d, int col0, const float* x) {
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    uint32_t b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) b[u] = pack_bf16x2(x[8 * g + 2 * u], x[8 * g + 2 * u + 1]);
    *reinterpret_cast<uint4*>(s_op + sw128_offset(d, col0 + 8 * g)) = make_uint4(b[0], b[1], b[2], b[3]);
  }
}

// 16 fp32 values (one thread's slice of a state row) to global memory.
__device__ __forceinline__ void store_slice(float* dst, const float* x) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int c = 0; c < 4; ++c) d4[c] = make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// kP1EvictFirst: phase-1 K and V loads under the L2 evict-first policy.
template <bool kP1EvictFirst>
__global__ void __launch_bounds__(kThreads, 1)
span_output_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const __grid_constant__ OutParams prm) {
  using L = OutSmem;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int H = prm.H;
  unsigned* err = prm.err;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  auto bar = [&](int slot) { return base + L::kBar + 8u * slot; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);

  // This CTA's set-up record: one round trip (the descriptors were uploaded
  // before the launch, but an L2 flush may have sent them back to DRAM).
  const int4* hd = reinterpret_cast<const int4*>(prm.heads + blockIdx.x);
  const int4 h0 = __ldg(hd), h1 = __ldg(hd + 1);
  const int i_begin = h0.x, n = h0.y, p1_begin = h0.z, n_p1 = h0.w;
  const int n1 = h1.x;         // phase-1 tiles
  const int n_first = h1.y;    // loads issued during the set-up
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(L::kFull + s), 1);
      mbar_init(bar(L::kEmpty + s), 2);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(L::kPReady + b), 1);
      mbar_init(bar(L::kPDone + b), kConvThreads);
      mbar_init(bar(L::kOReady + b), 1);
      mbar_init(bar(L::kPFree + b), 1);
      mbar_init(bar(L::kOFree + b), kGroupThreads);
      mbar_init(bar(L::kSSmem + b), kGroupThreads);
      mbar_init(bar(L::kDReady + b), 1);
      mbar_init(bar(L::kDFree + b), kGroupThreads);
      mbar_init(bar(L::kP1Ready + b), 1);
      mbar_init(bar(L::kP1Free + b), kGroupThreads);
    }
    mbar_init(bar(L::kP1Done), kGroupThreads);
    fence_mbar_init();
    // The first loads (phase-1 K and V, then the run's Q, K and V) go out
    // now, while the rest of the set-up completes; the stages are fresh.
    const int4 f0 = __ldg(hd + 2), f1 = __ldg(hd + 3);
    const int fr[2 * kFirstLoads] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
    const uint64_t pol = kP1EvictFirst ? l2_evict_first_policy() : 0;
#pragma unroll
    for (int u = 0; u < kFirstLoads; ++u) {
      if (u < n_first) {
        const uint32_t st = base + L::kStage0 + u * kStageBytes;
        const bool hint_kv = kP1EvictFirst && u < n1;
        if (u < n1) {
          mbar_arrive_expect_tx(bar(L::kFull + u), 2 * kRowTileBytes);
        } else {
          mbar_arrive_expect_tx(bar(L::kFull + u), kStageBytes);
          tma_load_3d(st + L::kQ, &tm_q, bar(L::kFull + u), 0, fr[2 * u], fr[2 * u + 1]);
        }
        if (hint_kv) {
          tma_load_3d_hint(st + L::kK, &tm_k, bar(L::kFull + u), 0, fr[2 * u], fr[2 * u + 1], pol);
          tma_load_3d_hint(st + L::kV, &tm_v, bar(L::kFull + u), 0, fr[2 * u], fr[2 * u + 1], pol);
        } else {
          tma_load_3d(st + L::kK, &tm_k, bar(L::kFull + u), 0, fr[2 * u], fr[2 * u + 1]);
          tma_load_3d(st + L::kV, &tm_v, bar(L::kFull + u), 0, fr[2 * u], fr[2 * u + 1]);
        }
      }
    }
    tma_prefetch_desc(&tm_o);
  }

  const WorkTile* list = prm.work + i_begin;
  const SpanDesc* p1 = prm.p1 + p1_begin;   // phase-1 pieces (one-launch pass only)
  int2* coord = reinterpret_cast<int2*>(smem + L::kCoord);
  SpanDesc* p1s = reinterpret_cast<SpanDesc*>(smem + L::kP1);
  // Warp 2 (the O issuer, idle until the set-up completes) stages the
  // producer's tile coordinates and the phase-1 pieces, at the same time as
  // thread 0 initialises the barriers and issues the first loads (behind
  // those, these small loads would wait for megabytes of tile traffic).
  if (warp == 2) {
    int2 c_lo = make_int2(0, 0), c_hi = make_int2(0, 0);
    if (lane < n) c_lo = make_int2(list[lane].row0, list[lane].head);
    if (lane + 32 < n && lane + 32 < kCoordSlots) c_hi = make_int2(list[lane + 32].row0, list[lane + 32].head);
    for (int j = lane; j < n_p1 && j < kP1Slots; j += 32) p1s[j] = p1[j];
    if (lane < n) coord[lane] = c_lo;
    if (lane + 32 < n && lane + 32 < kCoordSlots) coord[lane + 32] = c_hi;
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  auto p1_of = [&](int j) { return j < kP1Slots ? p1s[j] : p1[j]; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      const uint64_t pol = kP1EvictFirst ? l2_evict_first_policy() : 0;
      int u = 0;   // load index: phase-1 tiles, then the run's tiles
      for (int j = 0; j < n_p1 && ok; ++j) {
        const SpanDesc sd = p1_of(j);
        for (int r = 0; r < sd.len && ok; r += kTileRows, ++u) {
          if (u < n_first) continue;   // issued during the set-up
          const int s = u % kStages;
          if (!wait_or_flag(bar(L::kEmpty + s), ((u / kStages) & 1) ^ 1, err, kErrTimeoutMma)) { ok = false; break; }
          const uint32_t st = base + L::kStage0 + s * kStageBytes;
          mbar_arrive_expect_tx(bar(L::kFull + s), 2 * kRowTileBytes);
          if (kP1EvictFirst) {
            tma_load_3d_hint(st + L::kK, &tm_k, bar(L::kFull + s), 0, sd.row0 + r, sd.head, pol);
            tma_load_3d_hint(st + L::kV, &tm_v, bar(L::kFull + s), 0, sd.row0 + r, sd.head, pol);
          } else {
            tma_load_3d(st + L::kK, &tm_k, bar(L::kFull + s), 0, sd.row0 + r, sd.head);
            tma_load_3d(st + L::kV, &tm_v, bar(L::kFull + s), 0, sd.row0 + r, sd.head);
          }
        }
      }
      for (int i = 0; i < n && ok; ++i, ++u) {
        if (u < n_first) continue;   // issued during the set-up
        const int2 rc = i < kCoordSlots ? coord[i] : make_int2(list[i].row0, list[i].head);
        const int s = u % kStages;
        if (!wait_or_flag(bar(L::kEmpty + s), ((u / kStages) & 1) ^ 1, err, kErrTimeoutMma)) { ok = false; break; }
        const uint32_t st = base + L::kStage0 + s * kStageBytes;
        mbar_arrive_expect_tx(bar(L::kFull + s), kStageBytes);
        tma_load_3d(st + L::kQ, &tm_q, bar(L::kFull + s), 0, rc.x, rc.y);
        tma_load_3d(st + L::kK, &tm_k, bar(L::kFull + s), 0, rc.x, rc.y);
        tma_load_3d(st + L::kV, &tm_v, bar(L::kFull + s), 0, rc.x, rc.y);
      }
      // Wait (bounded) for the last loads to land before the CTA can exit.
      for (int w = (u > kStages ? u - kStages : 0); w < u; ++w)
        mbar_wait_bounded(bar(L::kFull + w % kStages), (w / kStages) & 1, ok ? kWaitLimitNs : 1000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ front issuer
    constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, 0, 0);
    constexpr uint32_t id_kv = idesc_bf16_f32(128, 64, 1, 1);
    bool ok = true;
    int u = 0;
    // Zero K and V rows past `rows` in a stage (they may hold anything, even
    // NaN, or rows of another segment).
    auto zero_tail = [&](uint32_t st, int rows) {
      if (rows >= kTileRows) return;
      uint8_t* vrow = smem + (st + L::kV - base);
      uint8_t* krow = smem + (st + L::kK - base);
      for (int q = rows * 8 + lane; q < kTileRows * 8; q += 32) {
        *reinterpret_cast<uint4*>(vrow + q * 16) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(krow + q * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
    };
    // Phase 1: K^T V summed over each piece into TMEM region j & 1.
    for (int j = 0; j < n_p1 && ok; ++j) {
      const SpanDesc sd = p1_of(j);
      const int b = j & 1;
      if (j >= 2) ok = wait_or_flag(bar(L::kP1Free + b), ((j - 2) >> 1) & 1, err, kErrTimeoutMma);
      if (!__all_sync(0xffffffffu, ok)) break;
      for (int r = 0; r < sd.len; r += kTileRows, ++u) {
        const int s = u % kStages;
        ok = wait_or_flag(bar(L::kFull + s), (u / kStages) & 1, err, kErrTimeoutTma);
        if (!__all_sync(0xffffffffu, ok)) break;
        const uint32_t st = base + L::kStage0 + s * kStageBytes;
        zero_tail(st, sd.len - r);
        __syncwarp();
        tc_fence_after_sync();
        if (lane == 0) {
          const uint32_t colD = b ? kColD1 : kColD0;
          for (int kk = 0; kk < kTileRows / 16; ++kk)
            mma_bf16(tmem + colD, smem_desc_sw128(st + L::kK + kk * 2048, 0, 1024),
                     smem_desc_sw128(st + L::kV + kk * 2048, kRowTileBytes, 1024), id_kv,
                     (r > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(L::kEmpty + s));
          mma_commit(bar(L::kEmpty + s));
          if (r + kTileRows >= sd.len) mma_commit(bar(L::kP1Ready + b));
        }
        __syncwarp();
      }
    }
    // The dS regions take the run's tiles once phase 1 has been read out.
    if (ok && n_p1 > 0) ok = wait_or_flag(bar(L::kP1Done), 0, err, kErrTimeoutMma);
    ok = __all_sync(0xffffffffu, ok);
    TileHead nxt = (ok && n > 0) ? load_head(list) : TileHead{};
    for (int i = 0; i < n && ok; ++i, ++u) {
      const TileHead r = nxt;
      if (i + 1 < n) nxt = load_head(list + i + 1);
      const int s = u % kStages, b = i & 1;
      if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kFull + s), (u / kStages) & 1, err, kErrTimeoutTma)))
        break;
      const uint32_t st = base + L::kStage0 + s * kStageBytes;
      // (A partial tile is the last of its piece: no state update reads its
      // tail, and a view-head's last tile sums only its own rows.)
      zero_tail(st, r.nrows);
      __syncwarp();
      // P buffer b is free once P V of tile i-2 (which read it) has completed.
      bool ok2 = true;
      if (i >= 2) ok2 = wait_or_flag(bar(L::kPFree + b), ((i - 2) >> 1) & 1, err, kErrTimeoutMma);
      if (!__all_sync(0xffffffffu, ok2)) break;
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
      if (i >= 2) ok2 = wait_or_flag(bar(L::kDFree + b), ((i - 2) >> 1) & 1, err, kErrTimeoutMma);
      if (!__all_sync(0xffffffffu, ok2)) break;
      tc_fence_after_sync();
      if (lane == 0) {
        if (!(r.flags & kTileLast) || (r.flags & kTileFinalOut)) {
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
    TileHead nxt = n > 0 ? load_head(list) : TileHead{};
    for (int i = 0; i < n; ++i) {
      const TileHead r = nxt;
      if (i + 1 < n) nxt = load_head(list + i + 1);
      const int u = n1 + i;
      const int s = u % kStages, b = i & 1;
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
        mma_commit(bar(L::kPFree + b));
      }
      __syncwarp();
      // S(i) staged: O(i) += Q S; release the stage.
      if (!__all_sync(0xffffffffu, wait_or_flag(bar(L::kSSmem + b), (i >> 1) & 1, err, kErrTimeoutMma)))
        break;
      tc_fence_after_sync();
      if (lane == 0) {
        if (has_state) {
          const uint32_t sop = base + L::kS + b * kSOpBytes;
          for (int kk = 0; kk < kHeadDim / 16; ++kk)
            mma_bf16(tmem + colO, smem_desc_sw128(st + L::kQ + kk * 32, 16, 1024),
                     smem_desc_sw128(sop + kk * 2048, kStateTileBytes, 1024), id_n64_b_mn, 1u);
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
    TileMask nxt = n > 0 ? load_mask(list) : TileMask{};
    for (int i = 0; i < n; ++i) {
      const TileMask r = nxt;
      if (i + 1 < n) nxt = load_mask(list + i + 1);
      const int b = i & 1;
      int seg_start = 0;
      if (r.nbound > 1) {
        const int nb = r.nbound < kInlineBounds ? r.nbound : kInlineBounds;
        for (int q = 1; q < nb; ++q) {
          const int sb = inline_bound(r.inl, q);
          if (sb <= row) seg_start = sb;
        }
        for (int q = kInlineBounds; q < r.nbound; ++q) {
          const int sb = prm.bounds[r.bound0 + q];
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
      // Two 32-column chunks in turn; chunk q's bf16 pairs go to columns
      // 16q .. 16q + 15 of the half, over scores already read (chunk 1's land
      // over columns 16 .. 31 of chunk 0).
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t pk[16];
        if (all_zero) {
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = 0u;
        } else {
          uint32_t r0[32];
          tmem_ld_32cols(tmem + lane_base + colP + 32 * q, r0);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int jj = c0 + 32 * q + 2 * c;
            float p0 = __uint_as_float(r0[2 * c]);
            float p1v = __uint_as_float(r0[2 * c + 1]);
            if (!all_kept) {
              p0 = (jj >= seg_start && jj <= hi_col) ? p0 : 0.f;
              p1v = (jj + 1 >= seg_start && jj + 1 <= hi_col) ? p1v : 0.f;
            }
            pk[c] = pack_bf16x2(p0, p1v);
          }
        }
        tmem_st_16cols(tmem + lane_base + colP + 16 * q, pk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kPDone + b));
    }
  } else {
    // ------------------------------------------------------------ state and output
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    const int pi = (warp - kStateWarp0) >> 2;     // which of the quarter's two warps
    const int row = quarter * 32 + lane;          // tile row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    // State work: lanes 0..63 and their copy in lanes 64..127 hold state rows
    // d = row & 63; the lower copy handles columns 0..31, the upper 32..63,
    // and the quarter's two warps take 16 of those each.
    const int d = row & 63, sh = row >> 6;
    const int col0 = 32 * sh + 16 * pi;           // this thread's state columns col0 .. col0 + 15
    const int64_t slice = static_cast<int64_t>(d) * kHeadDim + col0;   // offset in a state
    bool ok = true;

    // Phase 1: each piece's K^T V out of TMEM into its workspace slot; then
    // this CTA counts itself in the grid-wide counter.
    for (int j = 0; j < n_p1 && ok; ++j) {
      const SpanDesc sd = p1_of(j);
      const int b = j & 1;
      ok = __all_sync(0xffffffffu, wait_or_flag(bar(L::kP1Ready + b), (j >> 1) & 1, err, kErrTimeoutMma));
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t r0[16];
      tmem_ld_16cols(tmem + lane_base + (b ? kColD1 : kColD0) + col0, r0);
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kP1Free + b));
      store_slice(prm.ws + static_cast<int64_t>(sd.slot) * kStateFloats + slice,
                  reinterpret_cast<const float*>(r0));
    }
    if (n_p1 > 0) {
      mbar_arrive(bar(L::kP1Done));
      __threadfence();
      named_barrier_sync(kNamedStateBar, kGroupThreads);
      if (tid == kStateWarp0 * 32) atomicAdd(prm.counter, 1u);
    }
    // Wait (bounded) until every phase-1 CTA has counted itself, once, before
    // the first read of another CTA's slots.
    bool synced = !prm.fused;
    auto grid_sync = [&]() {
      if (synced) return;
      synced = true;
      if (tid == kStateWarp0 * 32) {
        const unsigned long long t0 = global_timer_ns();
        while (ld_acquire_gpu(prm.counter) < static_cast<unsigned>(prm.n_p1_ctas)) {
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrTimeoutMma);
            break;
          }
          __nanosleep(64);
        }
      }
      named_barrier_sync(kNamedStateBar, kGroupThreads);
    };

    // The running state (row d, columns col0 ..) in fp32.  tag_run names the
    // start state it holds while it is one (after the first tile of a
    // one-tile piece, or a view's final state); -1 once tiles have been added
    // to it.  A run of pieces with the same start state (the packed branch
    // tiles of one parent) loads it once, and each S operand remembers the
    // start state it holds, so that it is staged once per operand.
    float s_run[16];
    int64_t tag_run = -1, tag_op0 = -1, tag_op1 = -1;
    auto carry_tag = [&](int view, int head) -> int64_t {
      return (static_cast<int64_t>(1) << 62) | (static_cast<int64_t>(view) << 16) | head;
    };
    auto start_tag = [&](const TileState& r) -> int64_t {
      if (!(r.flags & kTileFirst) || !(r.flags & kTileHasInit)) return -1;
      if (r.flags & kTileCarry) return carry_tag(r.final_idx, r.head);
      return ((static_cast<int64_t>(r.stateA) + 1) << 40) ^ ((static_cast<int64_t>(r.a_n)) << 34) ^
             ((static_cast<int64_t>(r.stateB) + 1) << 16) ^ (static_cast<int64_t>(r.b_n) << 10) ^
             static_cast<int64_t>(r.head);
    };
    // Sum, in order, of the states of term A (a_n states a_rows heads apart)
    // and term B (b_n workspace slots) into s_run.  The group reads each
    // state coalesced (thread g of the group takes float4 number g + 256 c),
    // the sum goes through S operand t & 1 (free: its last reader was Q S of
    // tile t - 2), and each thread takes its slice back from there.  The
    // buffer index is XOR-swizzled on the half-row so that both sides are
    // free of bank conflicts.
    auto sum_start = [&](int t, const TileState& r) {
      const int g = tid - kStateWarp0 * 32;
      const int na = r.a_n, total = r.a_n + r.b_n;
      const float* pa =
          na > 0 ? prm.stateA + (static_cast<int64_t>(r.stateA) * prm.a_rows + (prm.a_rows > 1 ? r.head : 0)) *
                                    kStateFloats
                 : nullptr;
      const int64_t sa = static_cast<int64_t>(prm.a_rows) * kStateFloats;
      const float* pb = r.b_n > 0 ? prm.ws + static_cast<int64_t>(r.stateB) * kStateFloats : nullptr;
      auto src = [&](int k) -> const float4* {
        return reinterpret_cast<const float4*>(k < na ? pa + k * sa : pb + static_cast<int64_t>(k - na) * kStateFloats) + g;
      };
      float4 acc[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      auto add4 = [](float4& x, const float4 y) { x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w; };
      int k = 0;
      for (; k + 2 <= total; k += 2) {
        const float4* p0 = src(k);
        const float4* p1 = src(k + 1);
        float4 x[4], y[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) x[c] = __ldcg(p0 + kGroupThreads * c);
#pragma unroll
        for (int c = 0; c < 4; ++c) y[c] = __ldcg(p1 + kGroupThreads * c);
#pragma unroll
        for (int c = 0; c < 4; ++c) add4(acc[c], x[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) add4(acc[c], y[c]);
      }
      if (k < total) {
        const float4* p0 = src(k);
#pragma unroll
        for (int c = 0; c < 4; ++c) add4(acc[c], __ldcg(p0 + kGroupThreads * c));
      }
      float4* buf = reinterpret_cast<float4*>(smem + L::kS + (t & 1) * kSOpBytes);
      if (t & 1) tag_op1 = -1; else tag_op0 = -1;
      // The buffer holds two warps' O staging: their TMA stores must have
      // read it.
      if (lane == 0) bulk_wait_read_all();
      named_barrier_sync(kNamedStateBar, kGroupThreads);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int f = g + kGroupThreads * c, hr = f >> 3;
        buf[hr * 8 + ((f & 7) ^ ((hr >> 1) & 7))] = acc[c];
      }
      named_barrier_sync(kNamedStateBar, kGroupThreads);
      const int hr = 2 * d + sh;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 v4 = buf[hr * 8 + ((4 * pi + c) ^ ((hr >> 1) & 7))];
        s_run[4 * c] = v4.x; s_run[4 * c + 1] = v4.y; s_run[4 * c + 2] = v4.z; s_run[4 * c + 3] = v4.w;
      }
      named_barrier_sync(kNamedStateBar, kGroupThreads);
    };
    // The running state becomes the start state of the piece starting at `r`
    // (its S is staged next into operand t & 1): zero, the final state this
    // CTA computed (carry), the one it holds already, or the sum of term A
    // and term B.
    auto start_piece = [&](int t, const TileState& r) {
      if (!(r.flags & kTileHasInit)) {
#pragma unroll
        for (int e = 0; e < 16; ++e) s_run[e] = 0.f;
        tag_run = -1;
        return;
      }
      const int64_t tag = start_tag(r);
      if (tag == tag_run) return;
      tag_run = tag;
      if (r.flags & kTileCarry) {
        // The running state has moved on since the view's last tile (a long
        // branch ran in between): this thread's own slice of the final
        // state, as it wrote it.
        const float4* p4 = reinterpret_cast<const float4*>(
            prm.final_out + (static_cast<int64_t>(r.final_idx) * H + r.head) * kStateFloats + slice);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 v4 = __ldcg(p4 + c);
          s_run[4 * c] = v4.x; s_run[4 * c + 1] = v4.y; s_run[4 * c + 2] = v4.z; s_run[4 * c + 3] = v4.w;
        }
        return;
      }
      if (prm.fused) grid_sync();
      sum_start(t, r);
    };

    // S(t) -> S operand t & 1 (when tile t uses a state and the operand does
    // not hold that start state already).  The operand was last read by Q S
    // of tile t-2, whose completion o_work(t-2) saw.
    auto stage = [&](int t, const TileState& r) {
      const int64_t tag = start_tag(r);
      const bool uses = !(r.flags & kTileFirst) || (r.flags & kTileHasInit);
      const int64_t held = (t & 1) ? tag_op1 : tag_op0;
      if (uses && !(tag >= 0 && tag == held)) {
        stage_state_slice(smem + L::kS + (t & 1) * kSOpBytes, d, col0, s_run);
        if (t & 1) tag_op1 = tag; else tag_op0 = tag;
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(L::kSSmem + (t & 1)));
    };

    // O(i) -> global (rows of the tile only), through this warp's O staging
    // when its 32 rows all lie in the tile (one TMA store), else row by row.
    bool o_pending = false;   // this warp's last TMA store may still read its staging
    auto o_work = [&](int i, const TileState& r, bool live) -> bool {
      const int b = i & 1;
      if (!live || !__all_sync(0xffffffffu, wait_or_flag(bar(L::kOReady + b), (i >> 1) & 1, err, kErrTimeoutMma)))
        return false;
      tc_fence_after_sync();
      const uint32_t colO = b ? kColO1 : kColO0;
      // The quarter's two warps take 32 of the 64 output columns each.  A
      // warp whose 32 rows all lie in the tile writes its 32 x 32 block,
      // 64-byte swizzled, into its O staging (once its previous store has
      // read it) and stores it with one TMA store; otherwise each thread
      // stores its own row if it lies in the tile.
      const bool whole = (quarter + 1) * 32 <= r.nrows;
      uint8_t* ob = smem + L::kS + (quarter >> 1) * kSOpBytes + kStateTileBytes + (quarter & 1) * kOQuarterBytes +
                    pi * (kOQuarterBytes / 2);
      if (whole && o_pending) {
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
      }
      uint4* dst = reinterpret_cast<uint4*>(
          prm.out + ((static_cast<int64_t>(r.row0) + row) * H + r.head) * kHeadDim + 32 * pi);
      const bool store = row < r.nrows;
      uint32_t r0[32];
      tmem_ld_32cols(tmem + lane_base + colO + 32 * pi, r0);
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kOFree + b));
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 v4 = make_uint4(pack_bf16x2(__uint_as_float(r0[8 * c]), __uint_as_float(r0[8 * c + 1])),
                                    pack_bf16x2(__uint_as_float(r0[8 * c + 2]), __uint_as_float(r0[8 * c + 3])),
                                    pack_bf16x2(__uint_as_float(r0[8 * c + 4]), __uint_as_float(r0[8 * c + 5])),
                                    pack_bf16x2(__uint_as_float(r0[8 * c + 6]), __uint_as_float(r0[8 * c + 7])));
        if (whole)
          *reinterpret_cast<uint4*>(ob + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) = v4;
        else if (store)
          dst[c] = v4;
      }
      if (whole) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tm_o, smem_addr(ob), 32 * pi, r.row0 + quarter * 32, r.head);
          bulk_commit_group();
        }
        o_pending = true;
      }
      return true;
    };

    // Tile i's dS into the running state; at the last tile of a view-head
    // that is the view's final state: write it out; the branch tiles of this
    // run that start from it (carry) find it in s_run.
    // (Without `live`, or when the wait runs out, nothing is read or
    // written, but the start-state tags change as they would have: they
    // decide which named barriers the group reaches.)
    auto take_ds = [&](int i, const TileState& r, bool live) -> bool {
      const int b = i & 1;
      const bool good =
          live && __all_sync(0xffffffffu, wait_or_flag(bar(L::kDReady + b), (i >> 1) & 1, err, kErrTimeoutMma));
      if (good) tc_fence_after_sync();
      if (!(r.flags & kTileLast) || (r.flags & kTileFinalOut)) {
        if (good) {
          uint32_t r0[16];
          tmem_ld_16cols(tmem + lane_base + (b ? kColD1 : kColD0) + col0, r0);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) s_run[e] += __uint_as_float(r0[e]);
        }
        tag_run = -1;
      }
      if (good) {
        tc_fence_before_sync();
        mbar_arrive(bar(L::kDFree + b));
      }
      if (r.flags & kTileFinalOut) {
        if (good)
          store_slice(prm.final_out + (static_cast<int64_t>(r.final_idx) * H + r.head) * kStateFloats + slice, s_run);
        tag_run = carry_tag(r.final_idx, r.head);
      }
      return good;
    };

    if (ok) griddep_wait();   // start states from the scan (three launches)
    // The group's named barriers (here, in the start-state sum and in the
    // grid-wide wait) are reached by all four warps alike: where they fall
    // depends on the tiles and the start-state tags only.  A warp whose
    // bounded wait ran out goes on through the loop without waiting, reading
    // or writing results (the error word is set; the pass is void).
    if (n > 0) {
      TileState cur = load_state(list);
      TileState nxt = n > 1 ? load_state(list + 1) : TileState{};
      start_piece(0, cur);
      stage(0, cur);
      for (int i = 0; i < n; ++i) {
        // S(i+1) first: the O issuer needs it right after P V of tile i+1.
        if (i + 1 < n || (cur.flags & kTileFinalOut)) ok = take_ds(i, cur, ok);
        if (i + 1 < n) {
          if (cur.flags & kTileLast) start_piece(i + 1, nxt);
          stage(i + 1, nxt);
        }
        ok = o_work(i, cur, ok);
        cur = nxt;
        if (i + 2 < n) nxt = load_state(list + i + 2);
      }
    }
    if (lane == 0) bulk_wait_all();   // the last O stores have completed
  }

  griddep_launch_dependents();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_span_output(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                               const CUtensorMap* tm_v, const CUtensorMap* tm_o, const SpanOutputArgs& a,
                               cudaStream_t stream) {
  if (a.grid <= 0) return cudaSuccess;
  const uint32_t bytes = OutSmem::kRequest;
  static std::atomic<uint64_t> done{0};
  auto kernel = a.p1_evict_first ? span_output_kernel<true> : span_output_kernel<false>;
  static std::atomic<uint64_t> done_hint{0};
  cudaError_t e = set_smem_limit_once(kernel, bytes, a.p1_evict_first ? done_hint : done);
  if (e != cudaSuccess) return e;
  OutParams p{};
  p.heads = a.heads;
  p.work = a.work;
  p.cta_begin = a.cta_begin;
  p.bounds = a.bounds;
  p.stateA = a.stateA;
  p.ws = a.ws;
  p.final_out = a.final_out;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.err = a.err;
  p.p1 = a.p1;
  p.p1_begin = a.p1_begin;
  p.counter = a.counter;
  p.a_rows = a.a_rows;
  p.H = a.H;
  p.fused = a.fused ? 1 : 0;
  p.n_p1_ctas = a.n_p1_ctas;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (a.fused) {
    // CTAs wait on one another: all of them must be resident at once.
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (a.fused || a.pdl) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, tm_q[0], tm_k[0], tm_v[0], *tm_o, p);
}

}  // namespace spanla
