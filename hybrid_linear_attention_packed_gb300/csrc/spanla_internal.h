// Internal interface between the host side of libspanla (validation,
// descriptor build, workspace, launches) and its CUDA kernels.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <vector>

namespace spanla {

constexpr int kHeadDim = 64;     // d_k = d_v
constexpr int kChunk = 64;       // rows per chunk of the state scan
constexpr int kTileRows = 128;   // rows per output tile (two chunks)
constexpr int kStateFloats = kHeadDim * kHeadDim;

// One 64-row chunk whose local state K_c^T V_c the chunk-state kernel
// computes.  Chunk i of the table owns state slot i of the workspace.
struct ChunkDesc {
  int32_t row0;   // first row of the chunk in the packed buffer
  int32_t len;    // valid rows, 1..64
};

// One run of state slots for the segmented scan: the slots of one segment
// (chunk mode: one slot per 64-row chunk and head, the grid's y index is the
// head) or of one segment-head (span mode: head >= 0, one slot per piece).
// The scan turns the run into exclusive prefixes in place and writes the
// run's total (the view's final state) to final_out[final_idx] when
// final_idx >= 0; a run of no slots gives the zero state.
struct ScanDesc {
  int32_t slot0;      // first state slot
  int32_t nslots;     // slots in the run (0 for an empty view)
  int32_t final_idx;  // index into the final-state output, or -1
  int32_t head;       // span mode: the head; chunk mode: -1 (all heads)
};

// One output tile of up to 128 rows, for one head (the grid's y index).
// Rows [row0, row0 + nrows) are contiguous; they hold one view's rows, one
// long branch's rows, or several whole short branches of the same parent.
// bounds[bound0 .. bound0 + nbound) are the ascending row offsets (relative to
// row0, first one 0) at which a segment starts inside the tile.  The tile's
// start state is  stateA[a] + stateB[b]  (a missing term is -1).
struct TileDesc {
  int32_t row0;
  int32_t nrows;
  int32_t stateA;   // parent view final state (pass) / cached state index
  int32_t stateB;   // exclusive chunk-prefix slot of the tile's first chunk
  int32_t bound0;
  int32_t nbound;
  int32_t pad0;
  int32_t pad1;
};

// bf16 path (span mode).  The output work -- every tile of every
// segment-head -- is laid out request by request (a view's tiles, then the
// tiles of the branches whose parent it is, head by head) and cut into one
// contiguous run per CTA of the output kernel, so that every CTA gets the
// same number of tiles.  A *piece* is the part of one segment-head (a view
// or a branch longer than one tile) inside one run.  Every piece of a view,
// and every piece of a long branch cut into two or more pieces, owns one
// state slot: the span-state kernel writes the piece's local sum K^T V
// there, and the scan turns the slots of each segment-head into exclusive
// prefixes, i.e. the state entering each piece.
struct SpanDesc {
  int32_t row0;   // first row of the piece
  int32_t len;    // rows in the piece (>= 1)
  int32_t head;
  int32_t slot;   // state slot (fp32 [64][64] at ws + slot * 4096)
};
static_assert(sizeof(SpanDesc) == 16, "SpanDesc layout");

// One tile of the span-output kernel's per-CTA schedule (64 bytes).  CTA c
// runs records [cta_begin[c], cta_begin[c+1]) in order: the tiles of its run.
// A piece's first tile loads the piece's start state, the sum of two runs of
// fp32 states:  term A = states stateA .. stateA + a_n - 1 of the A array
// (the parent view's final state: with three launches the final-state array,
// [n][H][64][64], a_n = 1; in the one-launch pass the parent view-head's
// piece states), and term B = slots stateB .. stateB + b_n - 1 of the
// workspace (the piece's own prefix: one scanned slot with three launches,
// the earlier pieces' states in the one-launch pass).  A piece flagged
// kTileCarry starts instead from the final state the same CTA computed at
// the last tile of the parent view-head (kTileFinalOut), which also writes it
// to the final-state output (view final_idx).  Every later tile of a piece
// continues from the state the previous one left.
constexpr int kInlineBounds = 16;
constexpr int32_t kTileFirst = 1;      // first tile of its piece: load the start state
constexpr int32_t kTileLast = 2;       // last tile of its piece: no state update
constexpr int32_t kTileHasInit = 4;    // the piece has a start state
constexpr int32_t kTileCarry = 8;      // start state: this CTA's last final state
constexpr int32_t kTileFinalOut = 16;  // last tile of a view-head: compute and write its final state
struct WorkTile {
  int32_t row0;
  int32_t nrows;
  int32_t head;
  int32_t flags;
  int32_t stateA;    // first state of term A (first tile of a piece)
  int32_t stateB;    // first slot of term B
  int32_t a_n;       // states in term A (0: none)
  int32_t b_n;       // slots in term B (0: none)
  int32_t final_idx; // view of a kTileFinalOut tile (else -1)
  int32_t bound0;    // segment starts in the global bounds table
  int32_t nbound;    // the first kInlineBounds are also inline below
  int32_t pad;
  uint8_t inl[kInlineBounds];
};
static_assert(sizeof(WorkTile) == 64, "WorkTile layout");

// Softmax-attention layer over the packed rows: one work item = up to 128
// query rows [r0, r0 + nrows) of one segment (or of several whole short
// branches of one parent) for one head (32 bytes).  Its keys, in processing
// order, are the prefix rows [ps, ps + pn) of the prefix arrays (the parent
// view of branch rows, visible to every query row), then own blocks of 128 rows starting at os,
// os + 128, ..., r0: all but the last are fully visible, and the last one is
// the tile itself, causal, where query row i sees key row j (both relative
// to r0) when seg_start(i) <= j <= i.  seg_start(i) is the largest entry of
// bounds[seg0 .. seg0 + nseg) not above i (0 when nseg = 0): the start of the
// packed branch that holds row i.
struct SaItem {
  int32_t r0;
  int32_t nrows;
  int32_t head;
  int32_t ps;
  int32_t pn;
  int32_t os;
  int32_t seg0;
  int32_t nseg;
};
static_assert(sizeof(SaItem) == 32, "SaItem layout");

// Host plan of a softmax layer: the items of every head, dealt to CTAs
// (CTA c runs items [cta_begin[c], cta_begin[c+1]) in that order).
struct SoftmaxPlan {
  std::vector<SaItem> items;
  std::vector<uint8_t> bounds;
  std::vector<int32_t> cta_begin;
  int grid = 0;
  int64_t key_blocks = 0;    // (query tile, 128-key block) products, all heads
};
// With branches_only, views get no tiles (their K and V are a prefix source
// only: branches over K and V kept from an earlier pass).
SoftmaxPlan make_softmax_plan(const int32_t* view_cu, int32_t V, const int32_t* branch_cu, int32_t B,
                              const int32_t* parent, int H, int max_ctas, bool branches_only = false);

// tm_pk / tm_pv: the arrays the items' prefix rows index (ps) -- the same as
// tm_k / tm_v within one pass.
cudaError_t launch_softmax_attn(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                const CUtensorMap* tm_v, const CUtensorMap* tm_pk,
                                const CUtensorMap* tm_pv, const SaItem* items,
                                const int32_t* cta_begin, int grid, const uint8_t* bounds,
                                float scale_log2e, float scale, void* out, float* lse, int H,
                                unsigned* err, cudaStream_t stream);

struct DeviceOperands {
  // TMA descriptors; [0] = bf16 value (or high part), [1] = low part (fp32 inputs).
  CUtensorMap q[2], k[2], v[2];
};

// Set the calling thread's last-error text (span_la_last_error_detail).
void set_last_error_detail(const char* text);

// Raise a kernel's dynamic shared-memory limit once per device (`done` holds
// one bit per device it was set on).
template <typename Kernel>
inline cudaError_t set_smem_limit_once(Kernel kernel, uint32_t bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Kernel launchers (each returns the launch error, if any).
cudaError_t launch_split_f32(const float* q, const float* k, const float* v, int64_t n,
                             void* hi_lo_base, cudaStream_t stream);

cudaError_t launch_chunk_state(bool split, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                               const ChunkDesc* chunks, int n_chunks, int H, float* ws,
                               unsigned* err, cudaStream_t stream, bool pdl);

// span_mode: one head per entry (ScanDesc::head); otherwise every entry
// covers all H heads (grid y).
cudaError_t launch_scan(const ScanDesc* scan, int n_scan, int H, bool span_mode, float* ws,
                        float* final_out, cudaStream_t stream, bool pdl);

// spans: the pieces in per-CTA order, CTA c running [span_begin[c], span_begin[c+1]).
// [prefetch, prefetch + prefetch_bytes) is brought into L2 on the way (the
// pass's descriptors; 16-byte aligned).
cudaError_t launch_span_state(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                              const SpanDesc* spans, const int32_t* span_begin, int grid,
                              float* ws, const void* prefetch, size_t prefetch_bytes, unsigned* err,
                              cudaStream_t stream);

// The output kernel's arguments.  For the one-launch pass (fused) each CTA
// first sums K^T V over its phase-1 pieces (p1[p1_begin[c] .. p1_begin[c+1]),
// slots of `ws`), then counts itself in *counter; a CTA that needs other
// CTAs' slots waits until *counter reaches n_p1_ctas (the CTAs with phase-1
// work).  The grid is then launched cooperatively (every CTA resident).
// One span-output CTA's set-up record, at a fixed stride, so that the CTA
// reads it in one round trip and its producer issues the first loads before
// the rest of the set-up: its tile records, its phase-1 pieces, its phase-1
// tiles (loads before the run's tiles) and the (row0, head) of its first
// kFirstLoads loads in load order (phase-1 K/V boxes first).
constexpr int kFirstLoads = 4;
// Phase-1 K and V bytes of a one-launch pass above which its phase-1 loads
// take the L2 evict-first policy.  Below it, the tiles' second read of K and
// V finds them in the 129 MB L2, and the policy would make it miss; above it
// that read misses anyway, and the policy spares the write-back of dirty
// lines that phase 1 would otherwise displace.
constexpr int64_t kP1EvictFirstBytes = 96ll << 20;

struct CtaHead {
  int32_t i_begin, n;          // tile records [i_begin, i_begin + n)
  int32_t p1_begin, n_p1;      // phase-1 pieces (one-launch pass)
  int32_t n1;                  // phase-1 tiles
  int32_t n_first;             // entries of `first`
  int32_t pad[2];
  int32_t first[2 * kFirstLoads];
};
static_assert(sizeof(CtaHead) == 64, "CtaHead is 64 bytes");

struct SpanOutputArgs {
  const CtaHead* heads = nullptr;
  const WorkTile* work = nullptr;
  const int32_t* cta_begin = nullptr;
  int grid = 0;
  const uint8_t* bounds = nullptr;
  const float* stateA = nullptr;   // term A array
  int a_rows = 1;                  // heads per state index of term A (H, or 1 for slots)
  float* ws = nullptr;             // slots (term B; phase-1 output)
  float* final_out = nullptr;      // view final states [V][H][64][64]
  void* out = nullptr;
  int H = 0;
  unsigned* err = nullptr;
  bool pdl = false;
  bool fused = false;
  const SpanDesc* p1 = nullptr;
  const int32_t* p1_begin = nullptr;
  unsigned* counter = nullptr;
  int n_p1_ctas = 0;
  bool p1_evict_first = false;     // phase-1 K, V loads under the L2 evict-first policy
};
// tm_q/k/v: 128-row boxes of one head; tm_o: the output array, 32-row boxes
// of one head (a warp's rows, stored with one TMA store when all lie in the
// tile).
cudaError_t launch_span_output(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                               const CUtensorMap* tm_v, const CUtensorMap* tm_o, const SpanOutputArgs& a,
                               cudaStream_t stream);

cudaError_t launch_tile_output(bool split, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                               const CUtensorMap* tm_v, const TileDesc* tiles, int n_tiles,
                               const uint8_t* bounds, const float* stateA, const float* stateB,
                               void* out, int H, unsigned* err, cudaStream_t stream, bool pdl);

cudaError_t launch_wait_timeout_probe(unsigned limit_us, unsigned* err, cudaStream_t stream);

// Fixed workspace of span_la_pass_noalloc (a file-scope device array).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
cudaError_t noalloc_scratch(uint8_t** scratch, unsigned** err);
// The error word of that path on the current device, or NULL when the path
// has not been set up on it (no lookup is made then).
cudaError_t noalloc_error_word(unsigned** err);

// Box sizes of the TMA descriptors each kernel expects.
constexpr int kChunkBoxRows = kChunk;     // chunk-state kernel: 64 rows x 2 heads
constexpr int kChunkBoxHeads = 2;
constexpr int kSpanBoxRows = 4 * kChunk;  // span-state kernel: 256 rows x 1 head
constexpr int kTileBoxRows = kTileRows;   // tile-output kernel: 128 rows x 1 head
constexpr int kOutStoreRows = 32;         // span-output kernel's O stores: 32 rows x 1 head

}  // namespace spanla
