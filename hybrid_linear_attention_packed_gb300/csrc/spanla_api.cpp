// Host side of libspanla: argument validation, the packed-pass descriptor
// build, the plan cache, the stream-ordered workspace, TMA descriptors and the
// launches, for the linear-attention pass and the softmax layer; also the
// diagnostics (status text, profiling counters, fault injection).
//
// A pass ("Serving 0.88M TPS from Two RTXs and Mac Minis", section "Kernels":
// one scan per pass, the small kernels fused) is enqueued, for bf16 inputs,
// as one cooperative launch of the span-output kernel (phase 1: the local
// states other SMs need; a grid-wide counter; then each SM sums the start
// states it needs and runs its output tiles, branch fork included), or, as
// the page lays it out, as span state -> segmented scan -> span output
// (span_la_pass_variant); for fp32 inputs as chunk state -> scan -> tile
// output.  Every launch covers the whole pass however many views and
// branches it holds, from descriptor tables built here from the host
// metadata.
// The softmax layer over the same rows is one launch (section "Softmax
// layer" below).
#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <mutex>
#include <queue>
#include <string>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "spanla.h"
#include "spanla_internal.h"

using namespace spanla;

namespace {

thread_local std::string g_detail;

span_la_status fail(span_la_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_detail = buf;
  return s;
}

span_la_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SPAN_LA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Structure of the bf16 pass (span_la_pass_variant): 0 = one launch, 1 =
// three launches (span state -> scan -> output).
std::atomic<int32_t> g_pass_variant{0};
bool one_launch() { return g_pass_variant.load(std::memory_order_relaxed) == 0; }

// Fault injection (span_la_fault_inject): the next g_fail_allocs device
// allocations of the library fail as if the device were out of memory.
std::atomic<int32_t> g_fail_allocs{0};

bool injected_alloc_failure() {
  int32_t n = g_fail_allocs.load(std::memory_order_relaxed);
  while (n > 0) {
    if (g_fail_allocs.compare_exchange_weak(n, n - 1, std::memory_order_relaxed)) return true;
  }
  return false;
}

// ------------------------------------------------------------------ per-device state
constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  bool supported = false;
  int num_sms = 1;
  unsigned* err = nullptr;   // device error word
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

span_la_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SPAN_LA_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    d.supported = (major == 10 && minor == 3);
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || d.num_sms < 1)
      d.num_sms = 1;
    if (!d.supported) {
      d.ready = true;
      return fail(SPAN_LA_ERR_UNSUPPORTED,
                  "libspanla is built for sm_103a only; device %d is sm_%d%d", dev, major, minor);
    }
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
        return fail(SPAN_LA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    unsigned* err = nullptr;
    e = cudaMalloc(&err, sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(error word)");
    e = cudaMemset(err, 0, sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(error word)");
    cudaMemPool_t pool;
    if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) {
      uint64_t keep = UINT64_MAX;   // keep freed workspace in the pool between calls
      cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    }
    d.err = err;
    d.ready = true;
  }
  if (!d.supported) return fail(SPAN_LA_ERR_UNSUPPORTED, "device %d is not sm_103", dev);
  *out = &d;
  return SPAN_LA_OK;
}

// ------------------------------------------------------------------ profiling
constexpr int kKernelSplit = 0, kKernelChunk = 1, kKernelScan = 2, kKernelTile = 3,
              kKernelSpanState = 4, kKernelSpanOutput = 5, kKernelSoftmax = 6;
const char* const kKernelNames[SPAN_LA_NUM_KERNELS] = {"split_f32", "chunk_state", "segmented_scan",
                                                       "tile_output", "span_state", "span_output",
                                                       "softmax_attn"};

std::atomic<int64_t> g_launches[SPAN_LA_NUM_KERNELS];
std::atomic<bool> g_profiling{false};

struct EventRecord {
  int kernel;
  cudaEvent_t start, stop;
};

std::mutex g_prof_mu;
std::vector<EventRecord> g_pending;
std::vector<cudaEvent_t> g_spare_events;
double g_ms[SPAN_LA_NUM_KERNELS];
int64_t g_timed[SPAN_LA_NUM_KERNELS];

cudaEvent_t take_event() {
  if (!g_spare_events.empty()) {
    cudaEvent_t e = g_spare_events.back();
    g_spare_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Launch through `fn`, counting it and (when profiling) timing it with events.
template <typename Fn>
cudaError_t counted_launch(int kernel, cudaStream_t stream, Fn&& fn) {
  EventRecord rec{kernel, nullptr, nullptr};
  const bool timing = g_profiling.load(std::memory_order_relaxed);
  if (timing) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    rec.start = take_event();
    rec.stop = take_event();
  }
  if (rec.start) cudaEventRecord(rec.start, stream);
  cudaError_t e = fn();
  if (e == cudaSuccess) g_launches[kernel].fetch_add(1, std::memory_order_relaxed);
  if (rec.start && rec.stop) {
    cudaEventRecord(rec.stop, stream);
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_pending.push_back(rec);
  }
  return e;
}

// Fold every pending event pair into the totals (caller holds g_prof_mu).
cudaError_t drain_events() {
  cudaError_t first = cudaSuccess;
  for (const EventRecord& r : g_pending) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (e == cudaSuccess) {
      g_ms[r.kernel] += ms;
      g_timed[r.kernel] += 1;
    } else if (first == cudaSuccess) {
      first = e;
    }
    g_spare_events.push_back(r.start);
    g_spare_events.push_back(r.stop);
  }
  g_pending.clear();
  return first;
}

// ------------------------------------------------------------------ validation
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

span_la_status check_dims(const span_la_dims& dims) {
  if (dims.head_dim != kHeadDim)
    return fail(SPAN_LA_ERR_UNSUPPORTED, "head_dim %d not supported (only 64)", dims.head_dim);
  if (dims.dtype != SPAN_LA_BF16 && dims.dtype != SPAN_LA_F32)
    return fail(SPAN_LA_ERR_UNSUPPORTED, "dtype %d not supported", dims.dtype);
  if (dims.num_heads < 1) return fail(SPAN_LA_ERR_INVALID, "num_heads %d < 1", dims.num_heads);
  if (dims.total_rows < 0 || dims.total_rows > INT32_MAX)
    return fail(SPAN_LA_ERR_INVALID, "total_rows %lld out of range", (long long)dims.total_rows);
  return SPAN_LA_OK;
}

struct Segment {
  int64_t start, end;
  int idx;   // >= 0 view index, < 0: -(branch + 1)
};

span_la_status check_cu(const int32_t* cu, int32_t n, int64_t T, const char* name,
                        std::vector<Segment>* segs, bool views) {
  if (n < 0) return fail(SPAN_LA_ERR_INVALID, "%s: negative count %d", name, n);
  if (n == 0) return SPAN_LA_OK;
  if (cu == nullptr) return fail(SPAN_LA_ERR_INVALID, "%s is NULL with count %d", name, n);
  for (int32_t s = 0; s < n; ++s) {
    if (cu[s] < 0 || cu[s + 1] < cu[s] || cu[s + 1] > T)
      return fail(SPAN_LA_ERR_INVALID, "%s[%d..%d] = %d..%d is not a non-decreasing range in [0, %lld]",
                  name, s, s + 1, cu[s], cu[s + 1], (long long)T);
    if (cu[s + 1] > cu[s]) segs->push_back({cu[s], cu[s + 1], views ? s : -(s + 1)});
  }
  return SPAN_LA_OK;
}

span_la_status check_overlap(std::vector<Segment>& segs) {
  std::sort(segs.begin(), segs.end(),
            [](const Segment& a, const Segment& b) { return a.start < b.start; });
  for (size_t s = 1; s < segs.size(); ++s)
    if (segs[s].start < segs[s - 1].end)
      return fail(SPAN_LA_ERR_INVALID, "segments overlap: rows [%lld, %lld) and [%lld, %lld)",
                  (long long)segs[s - 1].start, (long long)segs[s - 1].end,
                  (long long)segs[s].start, (long long)segs[s].end);
  return SPAN_LA_OK;
}

span_la_status check_parents(const int32_t* parent, int32_t B, int32_t n_parents) {
  if (B == 0) return SPAN_LA_OK;
  if (parent == nullptr) return fail(SPAN_LA_ERR_INVALID, "branch_parent is NULL");
  for (int32_t b = 0; b < B; ++b)
    if (parent[b] < 0 || parent[b] >= n_parents)
      return fail(SPAN_LA_ERR_INVALID, "branch_parent[%d] = %d not in [0, %d)", b, parent[b], n_parents);
  return SPAN_LA_OK;
}

// ------------------------------------------------------------------ descriptor build
// Two plans.
//  * span mode (bf16 inputs): every tile of every segment-head is laid out
//    request by request -- a view's tiles, then the tiles of the branches
//    whose parent it is, head by head -- and the sequence is cut into one
//    contiguous run per CTA of the output kernel, every run of the same
//    length (+-1 tile).  A piece (the part of one view-head or long-branch-head
//    inside one run) owns a state slot: span_state sums K^T V per piece, the
//    scan turns the slots of each segment-head into exclusive prefixes, and
//    span_output walks each run carrying the state across its pieces' tiles.
//    Short branches are packed (adjacent, contiguous, same parent) into
//    single tiles whose start state is the parent's final state.
//  * chunk mode (fp32 inputs, split in bf16 parts): one state per 64-row
//    chunk (chunk_state), the scan over chunks, and one CTA per 128-row tile
//    (tile_output) starting from its first chunk's prefix.
struct Plan {
  bool span_mode = true;
  std::vector<ScanDesc> scan;
  std::vector<uint8_t> bounds;
  // chunk mode
  std::vector<ChunkDesc> chunks;
  std::vector<TileDesc> tiles;
  // span mode
  std::vector<SpanDesc> spans;       // pieces, in span_state's per-CTA order
  std::vector<int32_t> span_begin;   // span_state CTA c runs spans[span_begin[c] .. span_begin[c+1])
  std::vector<WorkTile> work;        // span_output's runs, one after the other
  std::vector<int32_t> cta_begin;    // span_output CTA c runs work[cta_begin[c] .. cta_begin[c+1])
  int run_tiles = 0;                 // longest run (tiles)
  int64_t n_pieces = 0;              // output pieces (packed tiles included), all heads
  // one-launch pass: spans / span_begin are the phase-1 pieces per output CTA
  bool fused = false;
  int n_p1_ctas = 0;                 // CTAs with phase-1 pieces
  bool p1_evict_first = false;       // phase-1 loads under the L2 evict-first policy
  std::vector<int32_t> empty_views;  // views without rows (their final state is zero)

  int state_slots(int H) const {
    return span_mode ? static_cast<int>(spans.size()) : static_cast<int>(chunks.size()) * H;
  }
  int state_grid() const { return span_begin.empty() ? 0 : static_cast<int>(span_begin.size()) - 1; }
  int out_grid() const { return cta_begin.empty() ? 0 : static_cast<int>(cta_begin.size()) - 1; }
  size_t n_out_tiles() const { return span_mode ? work.size() : tiles.size(); }

  void push_bound(int32_t& bound0, int32_t& nbound) {
    bound0 = static_cast<int32_t>(bounds.size());
    nbound = 1;
    bounds.push_back(0);
  }

  // chunk mode: a segment (view: final_idx >= 0; long branch: stateA = parent).
  void add_chunk_segment(int64_t start, int64_t len, int final_idx, int stateA) {
    const int chunk0 = static_cast<int>(chunks.size());
    const int n = static_cast<int>((len + kChunk - 1) / kChunk);
    for (int c = 0; c < n; ++c) {
      const int64_t r = start + static_cast<int64_t>(c) * kChunk;
      chunks.push_back({static_cast<int32_t>(r), static_cast<int32_t>(std::min<int64_t>(kChunk, start + len - r))});
    }
    scan.push_back({chunk0, n, final_idx, -1});
    for (int64_t r = 0; r < len; r += kTileRows) {
      const int j = static_cast<int>(r / kTileRows);
      TileDesc t{};
      t.row0 = static_cast<int32_t>(start + r);
      t.nrows = static_cast<int32_t>(std::min<int64_t>(kTileRows, len - r));
      t.stateA = stateA;
      t.stateB = j == 0 ? -1 : chunk0 + 2 * j;
      push_bound(t.bound0, t.nbound);
      tiles.push_back(t);
    }
  }
};

// Branches in list order as output groups: short ones (<= 128 rows) packed
// greedily with adjacent, contiguous branches of the same parent into one
// tile (their segment starts go to the bounds table), longer ones alone.
struct BranchGroup {
  int parent;
  int64_t row0, len;
  bool is_long;
  int32_t bound0, nbound;
};

std::vector<BranchGroup> group_branches(const int32_t* cu, int32_t B, const int32_t* parent,
                                        std::vector<uint8_t>* bounds) {
  std::vector<BranchGroup> groups;
  int open = -1;   // short-branch group being filled
  for (int32_t b = 0; b < B; ++b) {
    const int64_t start = cu[b], len = cu[b + 1] - cu[b];
    if (len == 0) continue;
    if (len > kTileRows) {
      open = -1;
      groups.push_back({parent[b], start, len, true, 0, 1});
      continue;
    }
    if (open >= 0) {
      BranchGroup& g = groups[open];
      if (g.parent == parent[b] && g.row0 + g.len == start && g.len + len <= kTileRows) {
        bounds->push_back(static_cast<uint8_t>(g.len));
        g.nbound += 1;
        g.len += len;
        continue;
      }
    }
    BranchGroup g{parent[b], start, len, false, static_cast<int32_t>(bounds->size()), 1};
    bounds->push_back(0);
    open = static_cast<int>(groups.size());
    groups.push_back(g);
  }
  return groups;
}

Plan make_span_plan(const int32_t* view_cu, int32_t V, const int32_t* branch_cu, int32_t B,
                    const int32_t* parent, int H, int num_sms, bool fused) {
  Plan plan;
  plan.span_mode = true;
  const std::vector<BranchGroup> groups = group_branches(branch_cu, B, parent, &plan.bounds);

  // Requests in order: view p (when p < V) followed by the branch groups
  // whose parent is p.  Without views (branches from cached states) the
  // parents that occur, in increasing order.
  std::vector<int> gparents;
  for (const BranchGroup& g : groups) gparents.push_back(g.parent);
  std::sort(gparents.begin(), gparents.end());
  gparents.erase(std::unique(gparents.begin(), gparents.end()), gparents.end());
  std::vector<int> requests;
  for (int32_t v = 0; v < V; ++v) requests.push_back(v);
  for (int p : gparents)
    if (p >= V) requests.push_back(p);
  std::vector<std::vector<int>> by_parent_idx(requests.size());
  {
    std::vector<int> pos(requests.size());
    for (size_t r = 0; r < requests.size(); ++r) pos[r] = static_cast<int>(r);
    // requests are sorted (views 0..V-1, then parents >= V ascending)
    for (size_t g = 0; g < groups.size(); ++g) {
      const auto it = std::lower_bound(requests.begin(), requests.end(), groups[g].parent);
      by_parent_idx[it - requests.begin()].push_back(static_cast<int>(g));
    }
  }

  // Segment-head blocks, head-major: every head has the same sequence
  // (request by request: the view's tiles, then its branches' tiles).
  struct Block {
    int kind;      // 0 view, 1 long branch group, 2 packed short branches
    int id;        // view index or group index
    int head;
    int64_t row0, len;
    int ntiles;
  };
  // The blocks of head 0 first; the other heads repeat them.
  std::vector<Block> blocks;
  blocks.reserve(static_cast<size_t>(H) * (V + groups.size()));
  int64_t W0 = 0;
  for (size_t r = 0; r < requests.size(); ++r) {
    const int p = requests[r];
    if (p < V) {
      const int64_t len = view_cu[p + 1] - view_cu[p];
      const int nt = static_cast<int>((len + kTileRows - 1) / kTileRows);
      blocks.push_back({0, p, 0, view_cu[p], len, nt});
      W0 += nt;
    }
    for (int g : by_parent_idx[r]) {
      const BranchGroup& bg = groups[g];
      const int nt = bg.is_long ? static_cast<int>((bg.len + kTileRows - 1) / kTileRows) : 1;
      blocks.push_back({bg.is_long ? 1 : 2, g, 0, bg.row0, bg.len, nt});
      W0 += nt;
    }
  }
  const int64_t W = W0 * H;

  // Runs.  Every head has the same sequence of tiles, so when the SMs can
  // be split evenly over the heads, each head's sequence is cut into R equal
  // runs and run (p, h) goes to CTA p H + h: CTAs that start together read
  // the same rows of every head (the same DRAM pages).  Otherwise the whole
  // head-major sequence is cut into one run per SM.  Either way CTA c takes
  // the global tiles [cut(c), cut(c+1)) of a list ordered by CTA.
  const int64_t per_head = H > 0 ? W / H : 0;
  const int sms = std::max(1, num_sms);
  const int R = H > 0 ? sms / H : 0;
  const bool aligned = R >= 1 && per_head > 0 && static_cast<int64_t>(R) * H * 100 >= static_cast<int64_t>(sms) * 85;
  const int Rh = aligned ? static_cast<int>(std::min<int64_t>(R, per_head)) : 0;
  const int grid = aligned ? Rh * H : static_cast<int>(std::min<int64_t>(W, sms));
  // With runs aligned to heads, run (p, h) is run (p, 0) with the head (and
  // the slots) shifted: passes 1 and 2 below plan head 0 only, and its
  // records are repeated for the other heads afterwards.  Otherwise every
  // head's blocks are planned.
  const bool per_head_copy = aligned && H > 1;
  if (!per_head_copy) {
    const size_t n0 = blocks.size();
    for (int h = 1; h < H; ++h)
      for (size_t i = 0; i < n0; ++i) {
        blocks.push_back(blocks[i]);
        blocks.back().head = h;
      }
  }
  // start of CTA c's run in the head-major sequence, and its length
  auto run_start = [&](int c) -> int64_t {
    if (!aligned) return grid > 0 ? static_cast<int64_t>(c) * W / grid : 0;
    const int p = c / H, h = c % H;
    return static_cast<int64_t>(h) * per_head + static_cast<int64_t>(p) * per_head / Rh;
  };
  auto run_len = [&](int c) -> int64_t {
    if (!aligned) return run_start(c + 1) - run_start(c);
    const int p = c / H;
    return static_cast<int64_t>(p + 1) * per_head / Rh - static_cast<int64_t>(p) * per_head / Rh;
  };
  // CTA owning head-major tile g, and the end of that CTA's run
  auto cta_of = [&](int64_t g) -> int {
    if (!aligned) {
      int c = static_cast<int>(g * grid / W);
      while (c + 1 < grid && run_start(c + 1) <= g) ++c;
      while (c > 0 && run_start(c) > g) --c;
      return c;
    }
    const int h = static_cast<int>(g / per_head);
    const int64_t j = g - static_cast<int64_t>(h) * per_head;
    int p = static_cast<int>(j * Rh / per_head);
    while (p + 1 < Rh && static_cast<int64_t>(p + 1) * per_head / Rh <= j) ++p;
    while (p > 0 && static_cast<int64_t>(p) * per_head / Rh > j) --p;
    return p * H + h;
  };
  plan.cta_begin.assign(grid + 1, 0);
  for (int c = 0; c < grid; ++c) {
    plan.cta_begin[c + 1] = plan.cta_begin[c] + static_cast<int32_t>(run_len(c));
    plan.run_tiles = std::max<int>(plan.run_tiles, static_cast<int>(run_len(c)));
  }
  plan.work.resize(W);

  // Pass 1: every block's pieces (split at the run boundaries), and for the
  // one-launch pass, per view-head, the run that holds its last tile and
  // whether any tile of its branches lies in another run (then every piece
  // of the view, the last one too, publishes its state).
  struct BPiece { int j0, j1, c; };
  std::vector<BPiece> bps;
  bps.reserve(blocks.size() + grid);
  std::vector<int32_t> bp_off(blocks.size() + 1, 0);
  std::vector<int32_t> vlast(fused ? static_cast<size_t>(V) * H : 0, -1);
  std::vector<uint8_t> vall(fused ? static_cast<size_t>(V) * H : 0, 0);
  {
    int64_t g0 = 0;
    for (size_t bi = 0; bi < blocks.size(); ++bi) {
      const Block& bk = blocks[bi];
      bp_off[bi] = static_cast<int32_t>(bps.size());
      int64_t a0 = g0;
      const int64_t end = g0 + bk.ntiles;
      while (a0 < end) {
        const int c = cta_of(a0);
        const int64_t b0 = std::min<int64_t>(end, run_start(c) + run_len(c));
        bps.push_back({static_cast<int>(a0 - g0), static_cast<int>(b0 - g0), c});
        a0 = b0;
      }
      if (fused) {
        if (bk.kind == 0 && bk.ntiles > 0) vlast[static_cast<size_t>(bk.id) * H + bk.head] = bps.back().c;
        if (bk.kind != 0) {
          const size_t vh = static_cast<size_t>(groups[bk.id].parent) * H + bk.head;
          for (size_t q = bp_off[bi]; q < bps.size(); ++q)
            if (bps[q].c != vlast[vh]) vall[vh] = 1;
        }
      }
      g0 += bk.ntiles;
    }
    bp_off[blocks.size()] = static_cast<int32_t>(bps.size());
  }

  // Pass 2: state slots, start-state recipes and the tile records.
  std::vector<SpanDesc> pieces;   // pieces with a slot, in creation order
  std::vector<int> piece_cta;      // output CTA of each
  pieces.reserve(blocks.size() + grid);
  piece_cta.reserve(blocks.size() + grid);
  std::vector<int32_t> vslot0(fused ? static_cast<size_t>(V) * H : 0, 0);
  std::vector<int32_t> vnslot(fused ? static_cast<size_t>(V) * H : 0, 0);
  int64_t g0 = 0;
  for (size_t bi = 0; bi < blocks.size(); ++bi) {
    const Block& bk = blocks[bi];
    if (bk.kind == 0 && bk.ntiles == 0) {   // empty view: zero final state
      if (fused) {
        if (bk.head == 0) plan.empty_views.push_back(bk.id);
      } else {
        plan.scan.push_back({0, 0, bk.id, bk.head});
      }
      continue;
    }
    const int m = bp_off[bi + 1] - bp_off[bi];
    const BPiece* bp = bps.data() + bp_off[bi];
    const int32_t parent = bk.kind == 0 ? -1 : groups[bk.id].parent;
    const size_t pvh = parent >= 0 ? static_cast<size_t>(parent) * H + bk.head : 0;
    // pieces of this block that own a slot: k < nslots
    int nslots;
    if (!fused) nslots = (bk.kind == 0 || (bk.kind == 1 && m >= 2)) ? m : 0;
    else if (bk.kind == 0) nslots = vall[static_cast<size_t>(bk.id) * H + bk.head] ? m : m - 1;
    else nslots = bk.kind == 1 ? m - 1 : 0;
    const int slot0 = static_cast<int>(pieces.size());
    if (!fused && nslots > 0) plan.scan.push_back({slot0, nslots, bk.kind == 0 ? bk.id : -1, bk.head});
    if (fused && bk.kind == 0) {
      vslot0[static_cast<size_t>(bk.id) * H + bk.head] = slot0;
      vnslot[static_cast<size_t>(bk.id) * H + bk.head] = nslots;
    }
    for (int k = 0; k < m; ++k) {
      const int j0 = bp[k].j0, j1 = bp[k].j1, c = bp[k].c;
      if (k < nslots) {
        const int64_t r0 = bk.row0 + static_cast<int64_t>(j0) * kTileRows;
        const int64_t r1 = std::min<int64_t>(bk.row0 + bk.len, bk.row0 + static_cast<int64_t>(j1) * kTileRows);
        pieces.push_back({static_cast<int32_t>(r0), static_cast<int32_t>(r1 - r0), bk.head,
                          static_cast<int32_t>(pieces.size())});
        piece_cta.push_back(c);
      }
      ++plan.n_pieces;
      WorkTile w{};
      w.head = bk.head;
      w.final_idx = -1;
      w.stateA = -1;
      w.stateB = -1;
      int32_t init = 0;
      if (!fused) {
        // three launches: the parent's final state (scan output) and the
        // piece's scanned prefix slot
        if (parent >= 0) { w.stateA = parent; w.a_n = 1; }
        if (nslots > 0 && k > 0) { w.stateB = slot0 + k; w.b_n = 1; }
        init = (w.a_n + w.b_n) > 0 ? kTileHasInit : 0;
      } else {
        // one launch: the parent's final state from this CTA (carry) or as
        // the sum of the parent view-head's pieces; the own prefix as the
        // sum of the earlier pieces
        if (parent >= 0) {
          if (k == 0 && c == vlast[pvh]) {
            init = kTileHasInit | kTileCarry;
            w.final_idx = parent;
          } else if (vnslot[pvh] > 0) {
            w.stateA = vslot0[pvh];
            w.a_n = vnslot[pvh];
          }
        }
        if (k > 0) {
          w.stateB = slot0;
          w.b_n = k;
        }
        if (w.a_n + w.b_n > 0) init |= kTileHasInit;
      }
      if (bk.kind == 2) {
        const BranchGroup& bg = groups[bk.id];
        w.bound0 = bg.bound0;
        w.nbound = bg.nbound;
        for (int q = 0; q < kInlineBounds && q < bg.nbound; ++q) w.inl[q] = plan.bounds[bg.bound0 + q];
      } else {
        w.bound0 = 0;
        w.nbound = 1;
      }
      // CTA c's run is contiguous in the head-major order
      WorkTile* dst = plan.work.data() + plan.cta_begin[c] + (g0 + j0 - run_start(c));
      for (int j = j0; j < j1; ++j) {
        const int64_t r = static_cast<int64_t>(j) * kTileRows;
        w.row0 = static_cast<int32_t>(bk.row0 + r);
        w.nrows = static_cast<int32_t>(std::min<int64_t>(kTileRows, bk.len - r));
        w.flags = (j == j0 ? kTileFirst : 0) | (j + 1 == j1 ? kTileLast : 0) | init;
        if (fused && bk.kind == 0 && k + 1 == m && j + 1 == j1) {
          w.flags |= kTileFinalOut;
          w.final_idx = bk.id;
        }
        dst[j - j0] = w;
      }
    }
    g0 += bk.ntiles;
  }
  if (per_head_copy) {
    // Head h: the pieces, slots and scan entries of head 0 shifted by h
    // heads (slots are numbered head after head, S0 per head), and run
    // (p, h) a copy of run (p, 0) in CTA p H + h.
    const int32_t S0 = static_cast<int32_t>(pieces.size());
    const size_t n_scan0 = plan.scan.size();
    for (int h = 1; h < H; ++h) {
      for (int32_t u = 0; u < S0; ++u) {
        SpanDesc sd = pieces[u];
        sd.head = h;
        sd.slot += h * S0;
        pieces.push_back(sd);
        piece_cta.push_back(piece_cta[u] + h);
      }
      for (size_t e = 0; e < n_scan0; ++e) {
        ScanDesc sc = plan.scan[e];
        if (sc.nslots > 0) sc.slot0 += h * S0;
        sc.head = h;
        plan.scan.push_back(sc);
      }
    }
    for (int p = 0; p < Rh; ++p) {
      const WorkTile* src = plan.work.data() + plan.cta_begin[p * H];
      const int32_t n = plan.cta_begin[p * H + 1] - plan.cta_begin[p * H];
      for (int h = 1; h < H; ++h) {
        WorkTile* dst = plan.work.data() + plan.cta_begin[p * H + h];
        std::memcpy(dst, src, static_cast<size_t>(n) * sizeof(WorkTile));
        for (int32_t i = 0; i < n; ++i) {
          dst[i].head = h;
          // the parent's final state (three launches, or a carry) is not a slot
          if (fused && dst[i].stateA >= 0) dst[i].stateA += h * S0;
          if (dst[i].stateB >= 0) dst[i].stateB += h * S0;
        }
      }
    }
    plan.n_pieces *= H;
  }
  if (fused) {
    // phase-1 pieces listed per output CTA (index = the CTA of the run)
    plan.span_begin.assign(grid + 1, 0);
    for (int c : piece_cta) ++plan.span_begin[c + 1];
    for (int c = 0; c < grid; ++c) {
      plan.n_p1_ctas += plan.span_begin[c + 1] > 0;
      plan.span_begin[c + 1] += plan.span_begin[c];
    }
    plan.spans.resize(pieces.size());
    std::vector<int32_t> fill(plan.span_begin.begin(), plan.span_begin.end() - 1);
    int64_t p1_bytes = 0;
    for (size_t u = 0; u < pieces.size(); ++u) {
      plan.spans[fill[piece_cta[u]]++] = pieces[u];
      p1_bytes += static_cast<int64_t>(pieces[u].len) * 2 * kHeadDim * 2;
    }
    plan.p1_evict_first = p1_bytes > kP1EvictFirstBytes;
    plan.fused = true;
    return plan;
  }

  // span_state: with no more pieces than SMs, piece k goes to the CTA that
  // runs its output (rows read together stay together); otherwise the
  // pieces are dealt longest first onto the least-loaded CTA.
  const int64_t n_sp = static_cast<int64_t>(pieces.size());
  if (n_sp > 0) {
    std::vector<int32_t> owner(n_sp);   // span_state CTA of each piece
    int sgrid = 0;
    if (n_sp <= sms && grid <= sms) {
      // CTAs that have pieces, numbered in output-CTA order
      std::vector<int32_t> remap(grid, -1);
      for (int64_t u = 0; u < n_sp; ++u) remap[piece_cta[u]] = 1;
      for (int c = 0; c < grid; ++c) remap[c] = remap[c] > 0 ? sgrid++ : -1;
      for (int64_t u = 0; u < n_sp; ++u) owner[u] = remap[piece_cta[u]];
    } else {
      sgrid = static_cast<int>(std::min<int64_t>(n_sp, sms));
      std::vector<int64_t> order(n_sp);
      for (int64_t u = 0; u < n_sp; ++u) order[u] = u;
      std::stable_sort(order.begin(), order.end(),
                       [&](int64_t a, int64_t b) { return pieces[a].len > pieces[b].len; });
      using Slot = std::pair<int64_t, int>;   // (rows assigned, cta)
      std::vector<Slot> heap_store;
      heap_store.reserve(sgrid);
      std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap(std::greater<Slot>(),
                                                                          std::move(heap_store));
      for (int c = 0; c < sgrid; ++c) heap.push({0, c});
      for (int64_t u : order) {
        Slot sl = heap.top();
        heap.pop();
        owner[u] = sl.second;
        sl.first += pieces[u].len;
        heap.push(sl);
      }
    }
    // counting sort of the pieces by owner, keeping creation order within a CTA
    plan.span_begin.assign(sgrid + 1, 0);
    for (int64_t u = 0; u < n_sp; ++u) ++plan.span_begin[owner[u] + 1];
    for (int c = 0; c < sgrid; ++c) plan.span_begin[c + 1] += plan.span_begin[c];
    plan.spans.resize(n_sp);
    std::vector<int32_t> fill(plan.span_begin.begin(), plan.span_begin.end() - 1);
    for (int64_t u = 0; u < n_sp; ++u) plan.spans[fill[owner[u]]++] = pieces[u];
  }
  return plan;
}

Plan make_plan(const int32_t* view_cu, int32_t V, const int32_t* branch_cu, int32_t B,
               const int32_t* parent, int H, bool span_mode, int num_sms, bool fused = false) {
  if (span_mode) return make_span_plan(view_cu, V, branch_cu, B, parent, H, num_sms, fused && V > 0);
  Plan plan;
  plan.span_mode = false;
  for (int32_t s = 0; s < V; ++s)
    plan.add_chunk_segment(view_cu[s], view_cu[s + 1] - view_cu[s], s, -1);
  const std::vector<BranchGroup> groups = group_branches(branch_cu, B, parent, &plan.bounds);
  for (const BranchGroup& g : groups) {
    if (g.is_long) {
      plan.add_chunk_segment(g.row0, g.len, -1, g.parent);
    } else {
      TileDesc t{};
      t.row0 = static_cast<int32_t>(g.row0);
      t.nrows = static_cast<int32_t>(g.len);
      t.stateA = g.parent;
      t.stateB = -1;
      t.bound0 = g.bound0;
      t.nbound = g.nbound;
      plan.tiles.push_back(t);
    }
  }
  return plan;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

template <typename T>
size_t put(std::vector<uint8_t>& host, const std::vector<T>& v) {
  const size_t off = host.size();
  host.resize(align256(off + v.size() * sizeof(T)), 0);
  if (!v.empty()) std::memcpy(host.data() + off, v.data(), v.size() * sizeof(T));
  return off;
}

template <typename T>
size_t bytes_of(const std::vector<T>& v) { return align256(v.size() * sizeof(T)); }

// 3-D view (d, token, head) of a [T][H][64] bf16 array; box = {box_cols,
// rows, heads} (128-byte swizzle for 64 columns, 64-byte for 32).
span_la_status encode_map(CUtensorMap* map, const void* base, int64_t T, int H, int box_rows,
                          int box_heads, int box_cols = kHeadDim) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(T),
                              static_cast<cuuint64_t>(H)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(H) * kHeadDim * 2, kHeadDim * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows),
                             static_cast<cuuint32_t>(box_heads)};
  const cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_cols == kHeadDim ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPAN_LA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return SPAN_LA_OK;
}

// Descriptors of a plan: one block the kernels read, plus what the launches
// need to know about it.
struct DescBlock {
  std::vector<uint8_t> host;
  size_t off_scan = 0, off_bounds = 0, off_a = 0, off_b = 0, off_c = 0, off_d = 0, off_h = 0;
  int grid = 0;            // span_output CTAs (span mode)
  int state_grid = 0;      // span_state CTAs (span mode)
  int n_scan = 0, n_chunks = 0, n_tiles = 0;
  int64_t state_slots = 0; // 16 KiB fp32 states of the workspace (all heads)
  size_t n_out_tiles = 0;
  size_t block_bytes = 0;  // size of the descriptor block on the device
  bool span_mode = true;
  bool fused = false;      // one-launch pass (span mode)
  int n_p1_ctas = 0;
  bool p1_evict_first = false;
  std::vector<int32_t> empty_views;
};

DescBlock make_desc(const Plan& plan, int H) {
  DescBlock d;
  d.span_mode = plan.span_mode;
  d.host.reserve(bytes_of(plan.scan) + bytes_of(plan.bounds) + bytes_of(plan.spans) + bytes_of(plan.span_begin) +
                 bytes_of(plan.work) + bytes_of(plan.cta_begin) + bytes_of(plan.chunks) + bytes_of(plan.tiles));
  d.off_scan = put(d.host, plan.scan);
  d.off_bounds = put(d.host, plan.bounds);
  if (plan.span_mode) {
    d.off_a = put(d.host, plan.spans);
    d.off_d = put(d.host, plan.span_begin);
    d.off_b = put(d.host, plan.work);
    d.off_c = put(d.host, plan.cta_begin);
    d.grid = plan.out_grid();
    d.state_grid = plan.state_grid();
    // Output CTAs' set-up records (phase-1 pieces are per output CTA only in
    // the one-launch pass; in three launches `spans` belong to span_state).
    std::vector<CtaHead> heads(static_cast<size_t>(d.grid));
    for (int c = 0; c < d.grid; ++c) {
      CtaHead& h = heads[c];
      h = CtaHead{};
      h.i_begin = plan.cta_begin[c];
      h.n = plan.cta_begin[c + 1] - plan.cta_begin[c];
      if (plan.fused) {
        h.p1_begin = plan.span_begin[c];
        h.n_p1 = plan.span_begin[c + 1] - plan.span_begin[c];
      }
      for (int j = 0; j < h.n_p1; ++j) {
        const SpanDesc& sd = plan.spans[h.p1_begin + j];
        for (int32_t r = 0; r < sd.len; r += kTileRows, ++h.n1)
          if (h.n_first < kFirstLoads) {
            h.first[2 * h.n_first] = sd.row0 + r;
            h.first[2 * h.n_first + 1] = sd.head;
            ++h.n_first;
          }
      }
      for (int i = 0; i < h.n && h.n_first < kFirstLoads; ++i, ++h.n_first) {
        const WorkTile& w = plan.work[h.i_begin + i];
        h.first[2 * h.n_first] = w.row0;
        h.first[2 * h.n_first + 1] = w.head;
      }
    }
    d.off_h = put(d.host, heads);
  } else {
    d.off_a = put(d.host, plan.chunks);
    d.off_b = put(d.host, plan.tiles);
  }
  d.n_scan = static_cast<int>(plan.scan.size());
  d.n_chunks = static_cast<int>(plan.chunks.size());
  d.n_tiles = static_cast<int>(plan.tiles.size());
  d.state_slots = plan.state_slots(H);
  d.n_out_tiles = plan.n_out_tiles();
  d.block_bytes = d.host.size();
  d.fused = plan.fused;
  d.n_p1_ctas = plan.n_p1_ctas;
  d.p1_evict_first = plan.p1_evict_first;
  d.empty_views = plan.empty_views;
  return d;
}

// ------------------------------------------------------------------ graph capture
// A host-to-device copy recorded while a stream is captured into a CUDA graph
// reads its host source every time the graph is launched.  The descriptor
// bytes of such a call are therefore moved into this registry and kept for the
// life of the process (a few KB per captured call).
std::mutex g_graph_mu;
std::vector<std::unique_ptr<std::vector<uint8_t>>> g_graph_bytes;

// Copy `bytes` to device `dst` on `stream`; when the stream is being captured,
// the bytes are first moved to storage that outlives the graph.
cudaError_t upload_descriptors(void* dst, std::vector<uint8_t>&& bytes, bool capturing, cudaStream_t stream) {
  if (bytes.empty()) return cudaSuccess;
  if (!capturing) return cudaMemcpyAsync(dst, bytes.data(), bytes.size(), cudaMemcpyHostToDevice, stream);
  std::lock_guard<std::mutex> lock(g_graph_mu);
  g_graph_bytes.push_back(std::make_unique<std::vector<uint8_t>>(std::move(bytes)));
  const std::vector<uint8_t>& kept = *g_graph_bytes.back();
  return cudaMemcpyAsync(dst, kept.data(), kept.size(), cudaMemcpyHostToDevice, stream);
}

// ------------------------------------------------------------------ pinned staging
// Cached descriptor blocks go to the device through pinned host buffers: a
// copy from pageable memory makes the calling thread wait until the stream's
// earlier work has finished, which puts the whole queue ahead of the pass on
// the host's critical path.  A buffer is reused once the copy that read it has
// completed (one event per buffer), so the pool holds as many buffers as
// uploads in flight at once, up to kPinnedBufs per device; past that an upload
// waits for the oldest copy.
constexpr size_t kPinnedBufs = 16;
constexpr size_t kPinnedMinBytes = 64 << 10;
struct PinnedBuf {
  int device = -1;
  uint8_t* p = nullptr;
  size_t cap = 0;
  cudaEvent_t done = nullptr;   // recorded after the copy that read it
  uint64_t used = 0;
};
std::mutex g_pin_mu;
std::vector<PinnedBuf> g_pin;
uint64_t g_pin_clock = 0;

// True when the copy that last read `b` has completed.
bool pinned_free(const PinnedBuf& b) {
  const cudaError_t q = cudaEventQuery(b.done);
  if (q == cudaErrorNotReady) (void)cudaGetLastError();   // not an error: clear it
  return q == cudaSuccess;
}

cudaError_t upload_pinned(void* dst, const std::vector<uint8_t>& bytes, int device, cudaStream_t stream) {
  if (bytes.empty()) return cudaSuccess;
  const size_t n = bytes.size();
  std::lock_guard<std::mutex> lock(g_pin_mu);
  PinnedBuf* pick = nullptr;
  size_t mine = 0;
  for (auto& b : g_pin) {
    if (b.device != device) continue;
    ++mine;
    // the smallest free buffer that fits; an event is queried only for a
    // buffer that would be a better pick (each query costs host time)
    if (b.cap >= n && (pick == nullptr || b.cap < pick->cap) && pinned_free(b)) pick = &b;
  }
  cudaError_t e = cudaSuccess;
  if (pick == nullptr) {
    if (mine < kPinnedBufs) {
      PinnedBuf nb;
      nb.device = device;
      e = cudaEventCreateWithFlags(&nb.done, cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
      g_pin.push_back(nb);
      pick = &g_pin.back();
    } else {   // the least recently used buffer of this device, once its copy is done
      for (auto& b : g_pin)
        if (b.device == device && (pick == nullptr || b.used < pick->used)) pick = &b;
      e = cudaEventSynchronize(pick->done);
    }
    if (e == cudaSuccess && pick->cap < n) {
      if (pick->p != nullptr) cudaFreeHost(pick->p);
      pick->p = nullptr;
      pick->cap = 0;
      size_t cap = kPinnedMinBytes;
      while (cap < n) cap *= 2;
      e = cudaHostAlloc(reinterpret_cast<void**>(&pick->p), cap, cudaHostAllocPortable);
      if (e == cudaSuccess) pick->cap = cap;
    }
    if (e != cudaSuccess) return e;
  }
  std::memcpy(pick->p, bytes.data(), n);
  e = cudaMemcpyAsync(dst, pick->p, n, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaEventRecord(pick->done, stream);
  pick->used = ++g_pin_clock;
  return e;
}

// ------------------------------------------------------------------ plan cache
// Passes with the same metadata (every layer of a model step, for instance)
// reuse one uploaded descriptor block: the plan depends on the metadata, the
// head count, the dtype and the SM count only.  A block is a stream-ordered
// allocation uploaded on the calling stream; a call on another stream first
// waits for that upload.  At most kCacheEntries blocks are kept per device.
// Every call that reads a block records an event on its stream afterwards
// (one event per stream, at most kMaxReaders streams per block), so that
// evicting a block frees it in stream order behind its last reads, without
// synchronising the host.  Calls made while their stream is being captured
// into a graph bypass the cache.
constexpr int kCacheEntries = 16;
constexpr size_t kMaxReaders = 8;

struct CacheEntry {
  int device = -1;
  std::vector<int32_t> key;
  DescBlock desc;
  uint8_t* d_block = nullptr;
  cudaEvent_t uploaded = nullptr;
  cudaStream_t upload_stream = nullptr;
  std::vector<std::pair<cudaStream_t, cudaEvent_t>> readers;   // last read per stream
  bool sync_on_evict = false;   // a read could not be recorded: synchronise before freeing
  uint64_t last_use = 0;
};

// Events of the plan cache (upload and reader events), kept for reuse per
// device instead of being destroyed and created on every miss (guarded by
// g_cache_mu, like the cache).
std::vector<cudaEvent_t> g_cache_events[kMaxDevices];

cudaError_t take_cache_event(int device, cudaEvent_t* ev) {
  std::vector<cudaEvent_t>& spare = g_cache_events[device & (kMaxDevices - 1)];
  if (!spare.empty()) {
    *ev = spare.back();
    spare.pop_back();
    return cudaSuccess;
  }
  return cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
}

void give_cache_event(int device, cudaEvent_t ev) {
  if (ev != nullptr) g_cache_events[device & (kMaxDevices - 1)].push_back(ev);
}

// Records on `stream` that the launches just enqueued there read `en`'s
// block.  A new stream beyond kMaxReaders takes over the oldest reader: it
// first waits for that reader's event, so its own event covers both.
cudaError_t note_reader(CacheEntry& en, cudaStream_t stream) {
  for (auto& r : en.readers)
    if (r.first == stream) return cudaEventRecord(r.second, stream);
  if (en.readers.size() >= kMaxReaders) {
    auto& oldest = en.readers.front();
    cudaError_t e = cudaStreamWaitEvent(stream, oldest.second, 0);
    if (e != cudaSuccess) return e;
    oldest.first = stream;
    e = cudaEventRecord(oldest.second, stream);
    std::rotate(en.readers.begin(), en.readers.begin() + 1, en.readers.end());
    return e;
  }
  cudaEvent_t ev = nullptr;
  cudaError_t e = take_cache_event(en.device, &ev);
  if (e != cudaSuccess) return e;
  e = cudaEventRecord(ev, stream);
  if (e != cudaSuccess) {
    give_cache_event(en.device, ev);
    return e;
  }
  en.readers.emplace_back(stream, ev);
  return cudaSuccess;
}

// Frees `en`'s block on `stream` behind its upload and every recorded read.
// On failure the block is left allocated (and the entry is kept).
cudaError_t release_entry(CacheEntry& en, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  if (en.sync_on_evict) {
    e = cudaDeviceSynchronize();
  } else {
    // work already on `stream` is ordered before the free without a wait
    if (en.upload_stream != stream) e = cudaStreamWaitEvent(stream, en.uploaded, 0);
    for (const auto& r : en.readers)
      if (e == cudaSuccess && r.first != stream) e = cudaStreamWaitEvent(stream, r.second, 0);
  }
  if (e == cudaSuccess) e = cudaFreeAsync(en.d_block, stream);
  if (e != cudaSuccess) return e;
  for (const auto& r : en.readers) give_cache_event(en.device, r.second);
  give_cache_event(en.device, en.uploaded);
  return cudaSuccess;
}

std::mutex g_cache_mu;
std::vector<CacheEntry> g_cache;
uint64_t g_cache_clock = 0;

// The last bf16 call's TMA descriptors per device (guarded by g_cache_mu).
struct MapCache {
  bool valid = false;
  int device = -1;
  const void* q = nullptr;
  const void* k = nullptr;
  const void* v = nullptr;
  int64_t T = 0;
  int H = 0;
  bool span_mode = false;
  DeviceOperands tile_ops{}, chunk_ops{};
  const void* o = nullptr;     // output array of tm_o
  CUtensorMap tm_o{};
};
MapCache g_maps[kMaxDevices];

std::vector<int32_t> plan_key(int device, int dtype, int H, int from_state, int num_sms,
                              const int32_t* view_cu, int32_t V, const int32_t* branch_cu,
                              int32_t B, const int32_t* parent) {
  std::vector<int32_t> key = {device, dtype, H, from_state, num_sms, V, B};
  if (V > 0) key.insert(key.end(), view_cu, view_cu + V + 1);
  if (B > 0) {
    key.insert(key.end(), branch_cu, branch_cu + B + 1);
    key.insert(key.end(), parent, parent + B);
  }
  return key;
}

// Cache key of a span_la_pass plan.  span_la_plan_prepare uses the same key,
// so that a pass finds the plan prepared for its metadata.
std::vector<int32_t> pass_key(int device, const span_la_dims& dims, int num_sms, bool fused,
                              const int32_t* view_cu, int32_t V, const int32_t* branch_cu,
                              int32_t B, const int32_t* parent) {
  return plan_key(device, dims.dtype, dims.num_heads, fused ? 4 : 0, num_sms, view_cu, V, branch_cu, B,
                  parent);
}

// The device block for `key` (built by `build` on a miss), usable on `stream`.
// The caller holds g_cache_mu until its launches are enqueued and recorded
// with note_reader on `*entry`, so that no other call evicts the block (or
// moves the entry) meanwhile.
template <typename Build>
span_la_status cached_block(const std::vector<int32_t>& key, int device, cudaStream_t stream,
                            Build&& build, const DescBlock** desc, const uint8_t** block,
                            CacheEntry** entry) {
  for (CacheEntry& en : g_cache) {
    if (en.device == device && en.key == key) {
      if (en.upload_stream != stream) {
        cudaError_t e = cudaStreamWaitEvent(stream, en.uploaded, 0);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(descriptor upload)");
      }
      en.last_use = ++g_cache_clock;
      *desc = &en.desc;
      *block = en.d_block;
      *entry = &en;
      return SPAN_LA_OK;
    }
  }
  int on_device = 0;
  size_t victim = g_cache.size();
  for (size_t i = 0; i < g_cache.size(); ++i) {
    if (g_cache[i].device != device) continue;
    ++on_device;
    if (victim == g_cache.size() || g_cache[i].last_use < g_cache[victim].last_use) victim = i;
  }
  if (on_device >= kCacheEntries) {
    cudaError_t e = release_entry(g_cache[victim], stream);
    if (e != cudaSuccess) return cuda_fail(e, "plan cache eviction");
    g_cache.erase(g_cache.begin() + victim);
  }
  CacheEntry en;
  en.device = device;
  en.key = key;
  en.desc = build();
  const size_t bytes = std::max<size_t>(en.desc.host.size(), 256);
  if (injected_alloc_failure())
    return fail(SPAN_LA_ERR_NOMEM, "cudaMallocAsync(descriptors, %zu): injected failure", bytes);
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&en.d_block), bytes, stream);
  if (e != cudaSuccess)
    return fail(SPAN_LA_ERR_NOMEM, "cudaMallocAsync(descriptors, %zu): %s", bytes, cudaGetErrorString(e));
  e = upload_pinned(en.d_block, en.desc.host, device, stream);
  if (e == cudaSuccess) e = take_cache_event(device, &en.uploaded);
  if (e == cudaSuccess) e = cudaEventRecord(en.uploaded, stream);
  if (e != cudaSuccess) {
    give_cache_event(device, en.uploaded);
    cudaFreeAsync(en.d_block, stream);
    return cuda_fail(e, "descriptor upload");
  }
  en.upload_stream = stream;
  en.last_use = ++g_cache_clock;
  g_cache.push_back(std::move(en));
  *desc = &g_cache.back().desc;
  *block = g_cache.back().d_block;
  *entry = &g_cache.back();
  return SPAN_LA_OK;
}

// After a call's launches: record the read of its cached block on `stream`.
span_la_status finish_read(CacheEntry* entry, cudaStream_t stream, span_la_status st) {
  if (entry == nullptr) return st;
  const cudaError_t e = note_reader(*entry, stream);
  if (e == cudaSuccess) return st;
  entry->sync_on_evict = true;
  return st == SPAN_LA_OK ? cuda_fail(e, "cudaEventRecord(descriptor read)") : st;
}

// The launches of one pass over descriptors already on the device (`block`):
// for fp32 inputs the split into bf16 parts (into `parts`, six [T][H][64]
// arrays), then state kernel -> scan -> output kernel, chained with
// programmatic dependent launch.  `states` holds desc.state_slots fp32
// states.  With `mc` (the caller holds g_cache_mu) the TMA descriptors of
// bf16 operands are reused from the last call on the same arrays.
span_la_status enqueue_pass(const DescBlock& desc, const uint8_t* block, uint8_t* parts, float* states,
                            unsigned* counter, const void* q, const void* k, const void* v,
                            const span_la_dims& dims, const float* stateA, float* final_out, void* out,
                            unsigned* err, cudaStream_t stream, MapCache* mc, int device) {
  const int H = dims.num_heads;
  const int64_t T = dims.total_rows;
  const bool split = dims.dtype == SPAN_LA_F32;
  cudaError_t e = cudaSuccess;
  span_la_status st = SPAN_LA_OK;

  // bf16 operand arrays the kernels read through TMA: the inputs themselves,
  // or, for fp32 inputs, their bf16 high / low parts made by the split kernel.
  const size_t part_bytes = static_cast<size_t>(T) * H * kHeadDim * 2;
  const void* ops[3][2] = {{q, nullptr}, {k, nullptr}, {v, nullptr}};
  if (split) {
    for (int t = 0; t < 3; ++t)
      for (int p = 0; p < 2; ++p) ops[t][p] = parts + (2 * t + p) * part_bytes;
    e = counted_launch(kKernelSplit, stream, [&] {
      return launch_split_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                              static_cast<const float*>(v), T * H * kHeadDim, parts, stream);
    });
    if (e != cudaSuccess) return cuda_fail(e, "split kernel launch");
  }
  DeviceOperands tile_ops{}, chunk_ops{};
  const bool need_maps = desc.n_out_tiles > 0 || desc.state_slots > 0;   // implies T > 0
  const bool map_hit = mc != nullptr && !split && mc->valid && mc->device == device && mc->q == q &&
                       mc->k == k && mc->v == v && mc->T == T && mc->H == H && mc->span_mode == desc.span_mode;
  if (map_hit) {
    tile_ops = mc->tile_ops;
    chunk_ops = mc->chunk_ops;
  }
  for (int t = 0; t < 3 && st == SPAN_LA_OK && need_maps && !map_hit; ++t) {
    for (int p = 0; p < (split ? 2 : 1) && st == SPAN_LA_OK; ++p) {
      CUtensorMap* tm = t == 0 ? &tile_ops.q[p] : t == 1 ? &tile_ops.k[p] : &tile_ops.v[p];
      CUtensorMap* cm = t == 0 ? &chunk_ops.q[p] : t == 1 ? &chunk_ops.k[p] : &chunk_ops.v[p];
      st = encode_map(tm, ops[t][p], T, H, kTileBoxRows, 1);
      // K and V boxes of the state kernel: 64 rows of two heads (chunk
      // mode) or 256 rows of one head (span mode).
      if (st == SPAN_LA_OK && t > 0)
        st = desc.span_mode ? encode_map(cm, ops[t][p], T, H, kSpanBoxRows, 1)
                            : encode_map(cm, ops[t][p], T, H, kChunkBoxRows, kChunkBoxHeads);
    }
  }
  if (st != SPAN_LA_OK) return st;
  // The span-output kernel stores whole 32-row x 32-column blocks of O with
  // TMA (one per warp).
  CUtensorMap tm_o{};
  const bool span_out = desc.span_mode && desc.n_out_tiles > 0;
  if (span_out) {
    if (mc != nullptr && mc->valid && map_hit && mc->o == out) {
      tm_o = mc->tm_o;
    } else {
      st = encode_map(&tm_o, out, T, H, kOutStoreRows, 1, 32);
      if (st != SPAN_LA_OK) return st;
    }
  }
  if (mc != nullptr && !split && need_maps && !map_hit) {
    mc->valid = true;
    mc->device = device;
    mc->q = q;
    mc->k = k;
    mc->v = v;
    mc->T = T;
    mc->H = H;
    mc->span_mode = desc.span_mode;
    mc->tile_ops = tile_ops;
    mc->chunk_ops = chunk_ops;
    mc->o = nullptr;
  }
  if (mc != nullptr && span_out && mc->valid && !split) {
    mc->o = out;
    mc->tm_o = tm_o;
  }

  if (desc.fused) {
    // One launch: the counter of the CTAs' phase-1 states starts at zero;
    // views without rows get the zero final state.
    e = cudaMemsetAsync(counter, 0, sizeof(unsigned), stream);
    for (size_t j = 0; j < desc.empty_views.size() && e == cudaSuccess; ++j)
      e = cudaMemsetAsync(final_out + static_cast<int64_t>(desc.empty_views[j]) * H * kStateFloats, 0,
                          static_cast<size_t>(H) * kStateFloats * sizeof(float), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(pass counter)");
    if (desc.n_out_tiles > 0) {
      SpanOutputArgs a;
      a.heads = reinterpret_cast<const CtaHead*>(block + desc.off_h);
      a.work = reinterpret_cast<const WorkTile*>(block + desc.off_b);
      a.cta_begin = reinterpret_cast<const int32_t*>(block + desc.off_c);
      a.grid = desc.grid;
      a.bounds = block + desc.off_bounds;
      a.stateA = states;
      a.a_rows = 1;
      a.ws = states;
      a.final_out = final_out;
      a.out = out;
      a.H = H;
      a.err = err;
      a.fused = true;
      a.p1 = reinterpret_cast<const SpanDesc*>(block + desc.off_a);
      a.p1_begin = reinterpret_cast<const int32_t*>(block + desc.off_d);
      a.counter = counter;
      a.n_p1_ctas = desc.n_p1_ctas;
      a.p1_evict_first = desc.p1_evict_first;
      e = counted_launch(kKernelSpanOutput, stream, [&] {
        return launch_span_output(tile_ops.q, tile_ops.k, tile_ops.v, &tm_o, a, stream);
      });
      if (e != cudaSuccess) return cuda_fail(e, "one-launch pass");
    }
    return SPAN_LA_OK;
  }

  bool kernel_before = split;   // a kernel precedes the next launch in the stream
  if (desc.state_slots > 0) {
    e = desc.span_mode
            ? counted_launch(kKernelSpanState, stream, [&] {
                return launch_span_state(chunk_ops.k, chunk_ops.v,
                                         reinterpret_cast<const SpanDesc*>(block + desc.off_a),
                                         reinterpret_cast<const int32_t*>(block + desc.off_d),
                                         desc.state_grid, states, block, desc.block_bytes, err, stream);
              })
            : counted_launch(kKernelChunk, stream, [&] {
                return launch_chunk_state(split, chunk_ops.k, chunk_ops.v,
                                          reinterpret_cast<const ChunkDesc*>(block + desc.off_a),
                                          desc.n_chunks, H, states, err, stream, kernel_before);
              });
    if (e != cudaSuccess) return cuda_fail(e, "chunk/span-state launch");
    kernel_before = true;
  }
  if (desc.n_scan > 0) {
    const bool pdl = kernel_before;
    e = counted_launch(kKernelScan, stream, [&] {
      return launch_scan(reinterpret_cast<const ScanDesc*>(block + desc.off_scan), desc.n_scan, H,
                         desc.span_mode, states, final_out, stream, pdl);
    });
    if (e != cudaSuccess) return cuda_fail(e, "scan launch");
    kernel_before = true;
  }
  if (desc.n_out_tiles > 0) {
    const bool pdl = kernel_before;
    if (desc.span_mode) {
      SpanOutputArgs a;
      a.heads = reinterpret_cast<const CtaHead*>(block + desc.off_h);
      a.work = reinterpret_cast<const WorkTile*>(block + desc.off_b);
      a.cta_begin = reinterpret_cast<const int32_t*>(block + desc.off_c);
      a.grid = desc.grid;
      a.bounds = block + desc.off_bounds;
      a.stateA = stateA;
      a.a_rows = H;
      a.ws = states;
      a.final_out = final_out;
      a.out = out;
      a.H = H;
      a.err = err;
      a.pdl = pdl;
      e = counted_launch(kKernelSpanOutput, stream, [&] {
        return launch_span_output(tile_ops.q, tile_ops.k, tile_ops.v, &tm_o, a, stream);
      });
    } else {
      e = counted_launch(kKernelTile, stream, [&] {
        return launch_tile_output(split, tile_ops.q, tile_ops.k, tile_ops.v,
                                  reinterpret_cast<const TileDesc*>(block + desc.off_b), desc.n_tiles,
                                  block + desc.off_bounds, stateA, states, out, H, err, stream, pdl);
      });
    }
    if (e != cudaSuccess) return cuda_fail(e, "output launch");
  }
  return SPAN_LA_OK;
}

// Common tail of both entry points: descriptors (cached, or uploaded into the
// call's workspace while the stream is being captured), workspace, launches.
template <typename BuildPlan>
span_la_status run_plan(const std::vector<int32_t>& key, BuildPlan&& build_plan, const void* q,
                        const void* k, const void* v, const span_la_dims& dims, const float* stateA,
                        float* final_out, void* out, cudaStream_t stream, DeviceState* dev, int device) {
  const int H = dims.num_heads;
  const int64_t T = dims.total_rows;
  const bool split = dims.dtype == SPAN_LA_F32;

  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  const bool use_cache = cap == cudaStreamCaptureStatusNone;
  std::unique_lock<std::mutex> cache_lock(g_cache_mu, std::defer_lock);
  DescBlock local;
  const DescBlock* desc = nullptr;
  const uint8_t* block = nullptr;
  CacheEntry* entry = nullptr;
  span_la_status st = SPAN_LA_OK;
  if (use_cache) {
    cache_lock.lock();
    st = cached_block(key, device, stream, [&] { return make_desc(build_plan(), H); }, &desc,
                      &block, &entry);
    if (st != SPAN_LA_OK) return st;
  } else {
    local = make_desc(build_plan(), H);
    desc = &local;
  }
  if (desc->n_out_tiles == 0 && desc->n_scan == 0 && desc->empty_views.empty()) return SPAN_LA_OK;

  // Workspace: the descriptor block when it is not cached, the state slots
  // and, for fp32 inputs, the six bf16 part arrays.
  const size_t desc_bytes = use_cache ? 0 : align256(desc->host.size());
  const size_t off_states = desc_bytes;
  const size_t state_bytes = static_cast<size_t>(desc->state_slots) * kStateFloats * sizeof(float);
  const size_t off_counter = align256(off_states + state_bytes);
  const size_t off_parts = off_counter + 256;
  const size_t part_bytes = static_cast<size_t>(T) * H * kHeadDim * 2;
  const size_t total = std::max<size_t>(off_parts + (split ? 6 * part_bytes : 0), 256);

  uint8_t* ws = nullptr;
  if (injected_alloc_failure()) return fail(SPAN_LA_ERR_NOMEM, "cudaMallocAsync(%zu): injected failure", total);
  e = cudaMallocAsync(reinterpret_cast<void**>(&ws), total, stream);
  if (e != cudaSuccess) return fail(SPAN_LA_ERR_NOMEM, "cudaMallocAsync(%zu): %s", total, cudaGetErrorString(e));
  if (!use_cache) {
    e = upload_descriptors(ws, std::move(local.host), true, stream);
    if (e != cudaSuccess) st = cuda_fail(e, "cudaMemcpyAsync(descriptors)");
    block = ws;
  }
  if (st == SPAN_LA_OK)
    st = enqueue_pass(*desc, block, ws + off_parts, reinterpret_cast<float*>(ws + off_states),
                      reinterpret_cast<unsigned*>(ws + off_counter), q, k, v, dims,
                      stateA, final_out, out, dev->err, stream,
                      use_cache ? &g_maps[device & (kMaxDevices - 1)] : nullptr, device);
  st = finish_read(entry, stream, st);
  cudaError_t ef = cudaFreeAsync(ws, stream);
  if (st == SPAN_LA_OK && ef != cudaSuccess) st = cuda_fail(ef, "cudaFreeAsync");
  return st;
}

// ------------------------------------------------------------------ softmax layer
// Descriptor block of a softmax-layer plan: items, CTA ranges, segment starts.
DescBlock make_softmax_desc(const SoftmaxPlan& plan) {
  DescBlock d;
  d.off_a = put(d.host, plan.items);
  d.off_c = put(d.host, plan.cta_begin);
  d.off_bounds = put(d.host, plan.bounds);
  d.grid = plan.grid;
  d.n_out_tiles = plan.items.size();
  return d;
}

// TMA descriptors of the last softmax call's operands per device (guarded by
// g_cache_mu).
struct SoftmaxMaps {
  bool valid = false;
  const void* q = nullptr;
  const void* k = nullptr;
  const void* v = nullptr;
  const void* pk = nullptr;
  const void* pv = nullptr;
  int64_t T = 0;
  int64_t prefix_rows = 0;
  int H = 0;
  DeviceOperands ops{};   // q[0], k[0], v[0]; prefix K in k[1], prefix V in v[1]
};
SoftmaxMaps g_sa_maps[kMaxDevices];

// One softmax-layer launch.  The items' prefix rows index pk / pv
// ([prefix_rows][H][64]): the pass's own k / v, or the K and V of views kept
// from an earlier pass (branches_only: the views get no tiles).
span_la_status run_softmax(const std::vector<int32_t>& key, const int32_t* view_cu, int32_t V,
                           const int32_t* branch_cu, int32_t B, const int32_t* parent, const void* q,
                           const void* k, const void* v, const void* pk, const void* pv, int64_t prefix_rows,
                           bool branches_only, const span_la_dims& dims, float scale, void* out, float* lse,
                           cudaStream_t stream, DeviceState* dev, int device) {
  const int H = dims.num_heads;
  const int64_t T = dims.total_rows;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  const bool use_cache = cap == cudaStreamCaptureStatusNone;
  auto build = [&] {
    return make_softmax_desc(make_softmax_plan(view_cu, V, branch_cu, B, parent, H, dev->num_sms, branches_only));
  };
  std::unique_lock<std::mutex> cache_lock(g_cache_mu, std::defer_lock);
  DescBlock local;
  const DescBlock* desc = nullptr;
  const uint8_t* block = nullptr;
  CacheEntry* entry = nullptr;
  span_la_status st = SPAN_LA_OK;
  if (use_cache) {
    cache_lock.lock();
    st = cached_block(key, device, stream, build, &desc, &block, &entry);
    if (st != SPAN_LA_OK) return st;
  } else {
    local = build();
    desc = &local;
  }
  if (desc->n_out_tiles == 0) return SPAN_LA_OK;

  uint8_t* ws = nullptr;
  if (!use_cache) {
    const size_t bytes = std::max<size_t>(desc->host.size(), 256);
    if (injected_alloc_failure()) return fail(SPAN_LA_ERR_NOMEM, "cudaMallocAsync(%zu): injected failure", bytes);
    e = cudaMallocAsync(reinterpret_cast<void**>(&ws), bytes, stream);
    if (e != cudaSuccess) return fail(SPAN_LA_ERR_NOMEM, "cudaMallocAsync(%zu): %s", bytes, cudaGetErrorString(e));
    e = upload_descriptors(ws, std::move(local.host), true, stream);
    if (e != cudaSuccess) st = cuda_fail(e, "cudaMemcpyAsync(descriptors)");
    block = ws;
  }
  if (st == SPAN_LA_OK) {
    DeviceOperands ops{};
    SoftmaxMaps& mc = g_sa_maps[device & (kMaxDevices - 1)];
    const bool hit = use_cache && mc.valid && mc.q == q && mc.k == k && mc.v == v && mc.pk == pk &&
                     mc.pv == pv && mc.T == T && mc.prefix_rows == prefix_rows && mc.H == H;
    if (hit) {
      ops = mc.ops;
    } else {
      st = encode_map(&ops.q[0], q, T, H, kTileBoxRows, 1);
      if (st == SPAN_LA_OK) st = encode_map(&ops.k[0], k, T, H, kTileBoxRows, 1);
      if (st == SPAN_LA_OK) st = encode_map(&ops.v[0], v, T, H, kTileBoxRows, 1);
      if (st == SPAN_LA_OK) {
        if (pk == k && pv == v && prefix_rows == T) {
          ops.k[1] = ops.k[0];
          ops.v[1] = ops.v[0];
        } else if (prefix_rows > 0) {
          st = encode_map(&ops.k[1], pk, prefix_rows, H, kTileBoxRows, 1);
          if (st == SPAN_LA_OK) st = encode_map(&ops.v[1], pv, prefix_rows, H, kTileBoxRows, 1);
        } else {
          // No prefix rows anywhere (every parent view is empty): never read.
          ops.k[1] = ops.k[0];
          ops.v[1] = ops.v[0];
        }
      }
      if (st == SPAN_LA_OK && use_cache) {
        mc.valid = true;
        mc.q = q;
        mc.k = k;
        mc.v = v;
        mc.pk = pk;
        mc.pv = pv;
        mc.T = T;
        mc.prefix_rows = prefix_rows;
        mc.H = H;
        mc.ops = ops;
      }
    }
    if (st == SPAN_LA_OK) {
      const float scale_log2e = scale * 1.4426950408889634f;
      e = counted_launch(kKernelSoftmax, stream, [&] {
        return launch_softmax_attn(ops.q, ops.k, ops.v, &ops.k[1], &ops.v[1],
                                   reinterpret_cast<const SaItem*>(block + desc->off_a),
                                   reinterpret_cast<const int32_t*>(block + desc->off_c), desc->grid,
                                   block + desc->off_bounds, scale_log2e, scale, out, lse, H, dev->err,
                                   stream);
      });
      if (e != cudaSuccess) st = cuda_fail(e, "softmax attention launch");
    }
  }
  st = finish_read(entry, stream, st);
  if (ws != nullptr) {
    cudaError_t ef = cudaFreeAsync(ws, stream);
    if (st == SPAN_LA_OK && ef != cudaSuccess) st = cuda_fail(ef, "cudaFreeAsync");
  }
  return st;
}

span_la_status check_operands(const void* q, const void* k, const void* v, void* out,
                              const span_la_dims& dims) {
  if (dims.total_rows == 0) return SPAN_LA_OK;
  if (!q || !k || !v || !out) return fail(SPAN_LA_ERR_INVALID, "q, k, v and out must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(SPAN_LA_ERR_INVALID, "q, k, v and out must be 16-byte aligned");
  return SPAN_LA_OK;
}

}  // namespace

namespace spanla {
void set_last_error_detail(const char* text) { g_detail = text; }
}  // namespace spanla

extern "C" {

span_la_status span_la_pass(const void* q, const void* k, const void* v, span_la_dims dims,
                            const int32_t* view_cu_seqlens, int32_t num_views,
                            const int32_t* branch_cu_seqlens, int32_t num_branches,
                            const int32_t* branch_parent, void* out, float* view_state_out,
                            cudaStream_t stream) {
  g_detail.clear();
  span_la_status st = check_dims(dims);
  if (st != SPAN_LA_OK) return st;
  std::vector<Segment> segs;
  if ((st = check_cu(view_cu_seqlens, num_views, dims.total_rows, "view_cu_seqlens", &segs, true)) != SPAN_LA_OK) return st;
  if ((st = check_cu(branch_cu_seqlens, num_branches, dims.total_rows, "branch_cu_seqlens", &segs, false)) != SPAN_LA_OK) return st;
  if ((st = check_overlap(segs)) != SPAN_LA_OK) return st;
  if ((st = check_parents(branch_parent, num_branches, num_views)) != SPAN_LA_OK) return st;
  if (!segs.empty() && (st = check_operands(q, k, v, out, dims)) != SPAN_LA_OK) return st;
  if (num_views > 0 && (view_state_out == nullptr || !aligned16(view_state_out)))
    return fail(SPAN_LA_ERR_INVALID, "view_state_out must be a non-NULL 16-byte aligned pointer");
  if (num_views == 0 && num_branches == 0) return SPAN_LA_OK;

  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != SPAN_LA_OK) return st;

  int device = 0;
  cudaGetDevice(&device);
  const bool fused = one_launch();
  const std::vector<int32_t> key = pass_key(device, dims, dev->num_sms, fused, view_cu_seqlens, num_views,
                                            branch_cu_seqlens, num_branches, branch_parent);
  auto build = [&] {
    return make_plan(view_cu_seqlens, num_views, branch_cu_seqlens, num_branches, branch_parent,
                     dims.num_heads, dims.dtype == SPAN_LA_BF16, dev->num_sms, fused);
  };
  return run_plan(key, build, q, k, v, dims, view_state_out, view_state_out, out, stream, dev, device);
}

span_la_status span_la_plan_prepare(span_la_dims dims, const int32_t* view_cu_seqlens, int32_t num_views,
                                    const int32_t* branch_cu_seqlens, int32_t num_branches,
                                    const int32_t* branch_parent, cudaStream_t stream) {
  g_detail.clear();
  span_la_status st = check_dims(dims);
  if (st != SPAN_LA_OK) return st;
  std::vector<Segment> segs;
  if ((st = check_cu(view_cu_seqlens, num_views, dims.total_rows, "view_cu_seqlens", &segs, true)) != SPAN_LA_OK) return st;
  if ((st = check_cu(branch_cu_seqlens, num_branches, dims.total_rows, "branch_cu_seqlens", &segs, false)) != SPAN_LA_OK) return st;
  if ((st = check_overlap(segs)) != SPAN_LA_OK) return st;
  if ((st = check_parents(branch_parent, num_branches, num_views)) != SPAN_LA_OK) return st;
  if (num_views == 0 && num_branches == 0) return SPAN_LA_OK;

  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != SPAN_LA_OK) return st;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cap != cudaStreamCaptureStatusNone)
    return fail(SPAN_LA_ERR_UNSUPPORTED, "span_la_plan_prepare: the stream is being captured (captured "
                                     "passes do not use the plan cache)");
  int device = 0;
  cudaGetDevice(&device);
  const bool fused = one_launch();
  const std::vector<int32_t> key = pass_key(device, dims, dev->num_sms, fused, view_cu_seqlens, num_views,
                                            branch_cu_seqlens, num_branches, branch_parent);
  auto build = [&] {
    return make_desc(make_plan(view_cu_seqlens, num_views, branch_cu_seqlens, num_branches, branch_parent,
                               dims.num_heads, dims.dtype == SPAN_LA_BF16, dev->num_sms, fused),
                     dims.num_heads);
  };
  std::lock_guard<std::mutex> lock(g_cache_mu);
  const DescBlock* desc = nullptr;
  const uint8_t* block = nullptr;
  CacheEntry* entry = nullptr;
  return cached_block(key, device, stream, build, &desc, &block, &entry);
}

span_la_status span_la_softmax_pass(const void* q, const void* k, const void* v, span_la_dims dims,
                                    const int32_t* view_cu_seqlens, int32_t num_views,
                                    const int32_t* branch_cu_seqlens, int32_t num_branches,
                                    const int32_t* branch_parent, float scale, void* out, float* lse_out,
                                    cudaStream_t stream) {
  g_detail.clear();
  span_la_status st = check_dims(dims);
  if (st != SPAN_LA_OK) return st;
  if (dims.dtype != SPAN_LA_BF16)
    return fail(SPAN_LA_ERR_UNSUPPORTED, "the softmax layer takes bf16 inputs only (dtype %d)", dims.dtype);
  if (!(scale >= 0.f) || !std::isfinite(scale))
    return fail(SPAN_LA_ERR_INVALID, "scale must be finite and >= 0 (0 selects 1/sqrt(head_dim))");
  if (scale == 0.f) scale = 1.f / std::sqrt(static_cast<float>(kHeadDim));
  std::vector<Segment> segs;
  if ((st = check_cu(view_cu_seqlens, num_views, dims.total_rows, "view_cu_seqlens", &segs, true)) != SPAN_LA_OK) return st;
  if ((st = check_cu(branch_cu_seqlens, num_branches, dims.total_rows, "branch_cu_seqlens", &segs, false)) != SPAN_LA_OK) return st;
  if ((st = check_overlap(segs)) != SPAN_LA_OK) return st;
  if ((st = check_parents(branch_parent, num_branches, num_views)) != SPAN_LA_OK) return st;
  if (!segs.empty() && (st = check_operands(q, k, v, out, dims)) != SPAN_LA_OK) return st;
  if (!segs.empty() && lse_out != nullptr && (reinterpret_cast<uintptr_t>(lse_out) & 3u) != 0)
    return fail(SPAN_LA_ERR_INVALID, "lse_out must be 4-byte aligned");
  if (segs.empty()) return SPAN_LA_OK;

  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != SPAN_LA_OK) return st;
  int device = 0;
  cudaGetDevice(&device);
  const std::vector<int32_t> key = plan_key(device, dims.dtype, dims.num_heads, 2, dev->num_sms, view_cu_seqlens,
                                            num_views, branch_cu_seqlens, num_branches, branch_parent);
  return run_softmax(key, view_cu_seqlens, num_views, branch_cu_seqlens, num_branches, branch_parent, q, k, v,
                     k, v, dims.total_rows, false, dims, scale, out, lse_out, stream, dev, device);
}

span_la_status span_la_softmax_branches_from_kv(const void* view_k, const void* view_v, int64_t view_rows,
                                                const int32_t* view_cu_seqlens, int32_t num_views,
                                                const void* q, const void* k, const void* v, span_la_dims dims,
                                                const int32_t* branch_cu_seqlens, int32_t num_branches,
                                                const int32_t* branch_parent, float scale, void* out,
                                                float* lse_out, cudaStream_t stream) {
  g_detail.clear();
  span_la_status st = check_dims(dims);
  if (st != SPAN_LA_OK) return st;
  if (dims.dtype != SPAN_LA_BF16)
    return fail(SPAN_LA_ERR_UNSUPPORTED, "the softmax layer takes bf16 inputs only (dtype %d)", dims.dtype);
  if (!(scale >= 0.f) || !std::isfinite(scale))
    return fail(SPAN_LA_ERR_INVALID, "scale must be finite and >= 0 (0 selects 1/sqrt(head_dim))");
  if (scale == 0.f) scale = 1.f / std::sqrt(static_cast<float>(kHeadDim));
  if (view_rows < 0 || view_rows > INT32_MAX) return fail(SPAN_LA_ERR_INVALID, "view_rows %lld out of range", (long long)view_rows);
  std::vector<Segment> vsegs, segs;
  if ((st = check_cu(view_cu_seqlens, num_views, view_rows, "view_cu_seqlens", &vsegs, true)) != SPAN_LA_OK) return st;
  if ((st = check_cu(branch_cu_seqlens, num_branches, dims.total_rows, "branch_cu_seqlens", &segs, false)) != SPAN_LA_OK) return st;
  if ((st = check_overlap(segs)) != SPAN_LA_OK) return st;
  if ((st = check_parents(branch_parent, num_branches, num_views)) != SPAN_LA_OK) return st;
  if (segs.empty()) return SPAN_LA_OK;
  if ((st = check_operands(q, k, v, out, dims)) != SPAN_LA_OK) return st;
  if (!vsegs.empty() && (view_k == nullptr || view_v == nullptr || !aligned16(view_k) || !aligned16(view_v)))
    return fail(SPAN_LA_ERR_INVALID, "view_k and view_v must be non-NULL and 16-byte aligned");
  if (lse_out != nullptr && (reinterpret_cast<uintptr_t>(lse_out) & 3u) != 0)
    return fail(SPAN_LA_ERR_INVALID, "lse_out must be 4-byte aligned");

  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != SPAN_LA_OK) return st;
  int device = 0;
  cudaGetDevice(&device);
  const std::vector<int32_t> key = plan_key(device, dims.dtype, dims.num_heads, 3, dev->num_sms, view_cu_seqlens,
                                            num_views, branch_cu_seqlens, num_branches, branch_parent);
  return run_softmax(key, view_cu_seqlens, num_views, branch_cu_seqlens, num_branches, branch_parent, q, k, v,
                     view_k, view_v, vsegs.empty() ? 0 : view_rows, true, dims, scale, out, lse_out, stream, dev,
                     device);
}

span_la_status span_la_branches_from_state(const float* cached_state, int32_t num_states,
                                           const void* q, const void* k, const void* v,
                                           span_la_dims dims, const int32_t* branch_cu_seqlens,
                                           int32_t num_branches, const int32_t* branch_parent,
                                           void* out, cudaStream_t stream) {
  g_detail.clear();
  span_la_status st = check_dims(dims);
  if (st != SPAN_LA_OK) return st;
  if (num_states < 0) return fail(SPAN_LA_ERR_INVALID, "num_states %d < 0", num_states);
  std::vector<Segment> segs;
  if ((st = check_cu(branch_cu_seqlens, num_branches, dims.total_rows, "branch_cu_seqlens", &segs, false)) != SPAN_LA_OK) return st;
  if ((st = check_overlap(segs)) != SPAN_LA_OK) return st;
  if ((st = check_parents(branch_parent, num_branches, num_states)) != SPAN_LA_OK) return st;
  if (!segs.empty() && (st = check_operands(q, k, v, out, dims)) != SPAN_LA_OK) return st;
  if (num_branches > 0 && (cached_state == nullptr || !aligned16(cached_state)))
    return fail(SPAN_LA_ERR_INVALID, "cached_state must be a non-NULL 16-byte aligned pointer");
  if (segs.empty()) return SPAN_LA_OK;

  DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != SPAN_LA_OK) return st;

  int device = 0;
  cudaGetDevice(&device);
  const std::vector<int32_t> key = plan_key(device, dims.dtype, dims.num_heads, 1, dev->num_sms, nullptr, 0,
                                            branch_cu_seqlens, num_branches, branch_parent);
  auto build = [&] {
    return make_plan(nullptr, 0, branch_cu_seqlens, num_branches, branch_parent, dims.num_heads,
                     dims.dtype == SPAN_LA_BF16, dev->num_sms);
  };
  return run_plan(key, build, q, k, v, dims, cached_state, nullptr, out, stream, dev, device);
}

span_la_status span_la_check(cudaStream_t stream) {
  g_detail.clear();
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  DeviceState* dev = nullptr;
  span_la_status st = device_state(&dev);
  if (st != SPAN_LA_OK) return st;
  unsigned word = 0;
  e = cudaMemcpy(&word, dev->err, sizeof(unsigned), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(error word)");
  if (word != 0) cudaMemset(dev->err, 0, sizeof(unsigned));
  // The no-allocation path's own error word, on a device where that path
  // (or its self-test) has run: read and cleared without allocating.
  unsigned na_word = 0;
  unsigned* na_err = nullptr;
  e = noalloc_error_word(&na_err);
  if (e != cudaSuccess) return cuda_fail(e, "no-allocation error word");
  if (na_err != nullptr) {
    e = cudaMemcpy(&na_word, na_err, sizeof(unsigned), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(no-allocation error word)");
    if (na_word != 0) {
      const unsigned zero = 0;
      e = cudaMemcpy(na_err, &zero, sizeof(unsigned), cudaMemcpyHostToDevice);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(clear no-allocation error word)");
    }
  }
  if (word != 0 || na_word != 0)
    return fail(SPAN_LA_ERR_TIMEOUT, "a bounded device wait ran out (error word 0x%x, no-allocation path 0x%x)",
                word, na_word);
  return SPAN_LA_OK;
}

const char* span_la_status_string(span_la_status s) {
  switch (s) {
    case SPAN_LA_OK: return "ok";
    case SPAN_LA_ERR_INVALID: return "invalid argument";
    case SPAN_LA_ERR_UNSUPPORTED: return "unsupported";
    case SPAN_LA_ERR_CUDA: return "CUDA error";
    case SPAN_LA_ERR_NOMEM: return "out of device memory";
    case SPAN_LA_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

const char* span_la_last_error_detail(void) { return g_detail.c_str(); }

int32_t span_la_version(void) { return 20000; }

span_la_status span_la_softmax_plan_stats(const int32_t* view_cu_seqlens, int32_t num_views,
                                          const int32_t* branch_cu_seqlens, int32_t num_branches,
                                          const int32_t* branch_parent, int32_t num_heads, int32_t num_sms,
                                          int64_t* stats) {
  g_detail.clear();
  if (stats == nullptr) return fail(SPAN_LA_ERR_INVALID, "stats is NULL");
  if (num_heads < 1) return fail(SPAN_LA_ERR_INVALID, "num_heads %d < 1", num_heads);
  if (num_sms < 1) return fail(SPAN_LA_ERR_INVALID, "num_sms %d < 1", num_sms);
  std::vector<Segment> segs;
  span_la_status st = SPAN_LA_OK;
  if ((st = check_cu(view_cu_seqlens, num_views, INT32_MAX, "view_cu_seqlens", &segs, true)) != SPAN_LA_OK) return st;
  if ((st = check_cu(branch_cu_seqlens, num_branches, INT32_MAX, "branch_cu_seqlens", &segs, false)) != SPAN_LA_OK) return st;
  if ((st = check_overlap(segs)) != SPAN_LA_OK) return st;
  if ((st = check_parents(branch_parent, num_branches, num_views)) != SPAN_LA_OK) return st;
  const SoftmaxPlan plan = make_softmax_plan(view_cu_seqlens, num_views, branch_cu_seqlens, num_branches,
                                             branch_parent, num_heads, num_sms);
  int64_t rows = 0;
  for (const SaItem& it : plan.items) rows += it.nrows;
  stats[0] = static_cast<int64_t>(plan.items.size());
  stats[1] = rows;
  stats[2] = plan.key_blocks;
  stats[3] = plan.grid;
  return SPAN_LA_OK;
}

span_la_status span_la_plan_stats(const int32_t* view_cu_seqlens, int32_t num_views,
                                  const int32_t* branch_cu_seqlens, int32_t num_branches,
                                  const int32_t* branch_parent, int32_t num_parents,
                                  int32_t from_state, int32_t num_heads, int32_t dtype,
                                  int32_t num_sms, int64_t* stats) {
  g_detail.clear();
  if (stats == nullptr) return fail(SPAN_LA_ERR_INVALID, "stats is NULL");
  if (num_heads < 1) return fail(SPAN_LA_ERR_INVALID, "num_heads %d < 1", num_heads);
  if (num_sms < 1) return fail(SPAN_LA_ERR_INVALID, "num_sms %d < 1", num_sms);
  if (dtype != SPAN_LA_BF16 && dtype != SPAN_LA_F32) return fail(SPAN_LA_ERR_UNSUPPORTED, "dtype %d", dtype);
  const int64_t T = INT32_MAX;
  std::vector<Segment> segs;
  span_la_status st = SPAN_LA_OK;
  if (from_state) num_views = 0;
  if ((st = check_cu(view_cu_seqlens, num_views, T, "view_cu_seqlens", &segs, true)) != SPAN_LA_OK) return st;
  if ((st = check_cu(branch_cu_seqlens, num_branches, T, "branch_cu_seqlens", &segs, false)) != SPAN_LA_OK) return st;
  if ((st = check_overlap(segs)) != SPAN_LA_OK) return st;
  if ((st = check_parents(branch_parent, num_branches, from_state ? num_parents : num_views)) != SPAN_LA_OK) return st;
  const int H = num_heads;
  const Plan plan = make_plan(view_cu_seqlens, num_views, branch_cu_seqlens, num_branches,
                              branch_parent, H, dtype == SPAN_LA_BF16, num_sms, !from_state && one_launch());
  // Every count is summed over heads.
  int64_t state_rows = 0, finals = 0, tile_rows = 0, state_reads = 0;
  for (const ChunkDesc& c : plan.chunks) state_rows += static_cast<int64_t>(c.len) * H;
  for (const SpanDesc& c : plan.spans) state_rows += c.len;
  for (const ScanDesc& s : plan.scan) finals += (s.final_idx >= 0) * (plan.span_mode ? 1 : H);
  if (plan.fused) finals = static_cast<int64_t>(num_views) * H;
  for (const TileDesc& t : plan.tiles) {
    tile_rows += static_cast<int64_t>(t.nrows) * H;
    state_reads += static_cast<int64_t>((t.stateA >= 0) + (t.stateB >= 0)) * H;
  }
  for (const WorkTile& w : plan.work) {
    tile_rows += w.nrows;
    if ((w.flags & kTileFirst) && !(w.flags & kTileCarry)) state_reads += w.a_n + w.b_n;
  }
  stats[0] = plan.state_slots(H);
  stats[1] = state_rows;
  stats[2] = static_cast<int64_t>(plan.scan.size()) * (plan.span_mode ? 1 : H);
  stats[3] = finals;
  stats[4] = static_cast<int64_t>(plan.n_out_tiles()) * (plan.span_mode ? 1 : H);
  stats[5] = tile_rows;
  stats[6] = state_reads;
  stats[7] = plan.span_mode ? plan.n_pieces : static_cast<int64_t>(plan.tiles.size()) * H;
  stats[8] = plan.span_mode ? plan.run_tiles : 1;
  return SPAN_LA_OK;
}

span_la_status span_la_profile_enable(int32_t enable) {
  g_profiling.store(enable != 0);
  return SPAN_LA_OK;
}

span_la_status span_la_profile_read(double* ms_total, int64_t* timed, int64_t* launches, int32_t n) {
  g_detail.clear();
  if (n < 0 || n > SPAN_LA_NUM_KERNELS) return fail(SPAN_LA_ERR_INVALID, "n %d not in [0, %d]", n, SPAN_LA_NUM_KERNELS);
  std::lock_guard<std::mutex> lock(g_prof_mu);
  cudaError_t e = drain_events();
  for (int k = 0; k < n; ++k) {
    if (ms_total) ms_total[k] = g_ms[k];
    if (timed) timed[k] = g_timed[k];
    if (launches) launches[k] = g_launches[k].load();
  }
  if (e != cudaSuccess) return cuda_fail(e, "profiling events");
  return SPAN_LA_OK;
}

span_la_status span_la_profile_reset(void) {
  g_detail.clear();
  std::lock_guard<std::mutex> lock(g_prof_mu);
  cudaError_t e = drain_events();
  for (int k = 0; k < SPAN_LA_NUM_KERNELS; ++k) {
    g_ms[k] = 0.0;
    g_timed[k] = 0;
    g_launches[k].store(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "profiling events");
  return SPAN_LA_OK;
}

const char* span_la_kernel_name(int32_t k) {
  return (k >= 0 && k < SPAN_LA_NUM_KERNELS) ? kKernelNames[k] : nullptr;
}

span_la_status span_la_pass_noalloc(const void* q, const void* k, const void* v, span_la_dims dims,
                                    const int32_t* view_cu_seqlens, int32_t num_views,
                                    const int32_t* branch_cu_seqlens, int32_t num_branches,
                                    const int32_t* branch_parent, void* out, float* view_state_out,
                                    cudaStream_t stream) {
  g_detail.clear();
  span_la_status st = check_dims(dims);
  if (st != SPAN_LA_OK) return st;
  if (dims.dtype != SPAN_LA_BF16)
    return fail(SPAN_LA_ERR_UNSUPPORTED,
                "span_la_pass_noalloc takes bf16 inputs only (fp32 inputs need per-call scratch "
                "for their bf16 parts; use span_la_pass)");
  std::vector<Segment> segs;
  if ((st = check_cu(view_cu_seqlens, num_views, dims.total_rows, "view_cu_seqlens", &segs, true)) != SPAN_LA_OK) return st;
  if ((st = check_cu(branch_cu_seqlens, num_branches, dims.total_rows, "branch_cu_seqlens", &segs, false)) != SPAN_LA_OK) return st;
  if ((st = check_overlap(segs)) != SPAN_LA_OK) return st;
  if ((st = check_parents(branch_parent, num_branches, num_views)) != SPAN_LA_OK) return st;
  if (!segs.empty() && (st = check_operands(q, k, v, out, dims)) != SPAN_LA_OK) return st;
  if (num_views > 0 && (view_state_out == nullptr || !aligned16(view_state_out)))
    return fail(SPAN_LA_ERR_INVALID, "view_state_out must be a non-NULL 16-byte aligned pointer");
  if (num_views == 0 && num_branches == 0) return SPAN_LA_OK;

  // Device checks without the allocating set-up of the other entry points.
  int dev = 0, major = 0, minor = 0, num_sms = 1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  if (!(major == 10 && minor == 3))
    return fail(SPAN_LA_ERR_UNSUPPORTED, "libspanla is built for sm_103a only; device %d is sm_%d%d",
                dev, major, minor);
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult qr;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr);
      if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || fn == nullptr)
        return fail(SPAN_LA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  uint8_t* ws = nullptr;
  unsigned* err = nullptr;
  e = noalloc_scratch(&ws, &err);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(fixed scratch)");

  // The same plan, descriptors and launches as span_la_pass (so the results
  // are the same bit for bit); the descriptors and the state slots live in
  // the fixed scratch.
  const int H = dims.num_heads;
  DescBlock desc = make_desc(make_plan(view_cu_seqlens, num_views, branch_cu_seqlens, num_branches,
                                       branch_parent, H, true, num_sms, one_launch()), H);
  const size_t off_states = align256(desc.host.size());
  const size_t off_counter = align256(off_states + static_cast<size_t>(desc.state_slots) * kStateFloats * sizeof(float));
  const size_t need = off_counter + sizeof(unsigned);
  if (need > kNoAllocScratchBytes)
    return fail(SPAN_LA_ERR_INVALID,
                "this pass needs %zu bytes of scratch; the fixed scratch of span_la_pass_noalloc holds "
                "%zu bytes (use span_la_pass)", need, kNoAllocScratchBytes);
  if (desc.n_out_tiles == 0 && desc.n_scan == 0 && desc.empty_views.empty()) return SPAN_LA_OK;

  // Everything the kernels read from the scratch is written by this call
  // first.  The error word is not cleared here: a wait that ran out stays
  // recorded until span_la_check reads it.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e == cudaSuccess) e = upload_descriptors(ws, std::move(desc.host), cap != cudaStreamCaptureStatusNone, stream);
  if (e != cudaSuccess) return cuda_fail(e, "descriptor upload");
  return enqueue_pass(desc, ws, nullptr, reinterpret_cast<float*>(ws + off_states),
                      reinterpret_cast<unsigned*>(ws + off_counter), q, k, v, dims,
                      view_state_out, view_state_out, out, err, stream, nullptr, dev);
}

span_la_status span_la_pass_variant(int32_t variant) {
  g_detail.clear();
  if (variant != SPAN_LA_PASS_ONE_LAUNCH && variant != SPAN_LA_PASS_THREE_LAUNCHES)
    return fail(SPAN_LA_ERR_INVALID, "unknown pass variant %d", variant);
  g_pass_variant.store(variant, std::memory_order_relaxed);
  return SPAN_LA_OK;
}

span_la_status span_la_fault_inject(int32_t kind, int32_t count) {
  g_detail.clear();
  if (kind != SPAN_LA_FAULT_ALLOC) return fail(SPAN_LA_ERR_INVALID, "unknown fault kind %d", kind);
  if (count < 0) return fail(SPAN_LA_ERR_INVALID, "count %d < 0", count);
  g_fail_allocs.store(count, std::memory_order_relaxed);
  return SPAN_LA_OK;
}

span_la_status span_la_selftest_wait_timeout_noalloc(int32_t limit_us, cudaStream_t stream) {
  g_detail.clear();
  if (limit_us < 1 || limit_us > 1000000)
    return fail(SPAN_LA_ERR_INVALID, "limit_us %d not in [1, 1000000]", limit_us);
  uint8_t* ws = nullptr;
  unsigned* err = nullptr;
  cudaError_t e = noalloc_scratch(&ws, &err);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-allocation error word)");
  e = launch_wait_timeout_probe(static_cast<unsigned>(limit_us), err, stream);
  if (e != cudaSuccess) return cuda_fail(e, "probe launch");
  return SPAN_LA_OK;
}

span_la_status span_la_selftest_wait_timeout(int32_t limit_us, cudaStream_t stream) {
  g_detail.clear();
  if (limit_us < 1 || limit_us > 1000000)
    return fail(SPAN_LA_ERR_INVALID, "limit_us %d not in [1, 1000000]", limit_us);
  DeviceState* dev = nullptr;
  span_la_status st = device_state(&dev);
  if (st != SPAN_LA_OK) return st;
  cudaError_t e = launch_wait_timeout_probe(static_cast<unsigned>(limit_us), dev->err, stream);
  if (e != cudaSuccess) return cuda_fail(e, "probe launch");
  return SPAN_LA_OK;
}

}  // extern "C"
