// Host side of libspanla: argument validation, the packed-pass descriptor
// build, the stream-ordered workspace, TMA descriptors and the launches.
//
// A pass ("Serving 0.88M TPS from Two RTXs and Mac Minis", section "Kernels":
// one scan per pass in three launches) is enqueued as
//   chunk-state  -> segmented scan -> tile output (view chunks + branch fork)
// over descriptor tables built here from the host metadata, so that each step
// is one launch for the whole pass however many views and branches it holds.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
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

// ------------------------------------------------------------------ per-device state
constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  bool supported = false;
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
struct Plan {
  std::vector<ChunkDesc> chunks;
  std::vector<ScanDesc> scan;
  std::vector<TileDesc> tiles;
  std::vector<uint8_t> bounds;

  // Chunk a segment for the scan; returns its first state slot.
  int add_chunks(int64_t start, int64_t len, int final_idx) {
    const int chunk0 = static_cast<int>(chunks.size());
    const int n = static_cast<int>((len + kChunk - 1) / kChunk);
    for (int c = 0; c < n; ++c) {
      const int64_t r = start + static_cast<int64_t>(c) * kChunk;
      chunks.push_back({static_cast<int32_t>(r), static_cast<int32_t>(std::min<int64_t>(kChunk, start + len - r))});
    }
    scan.push_back({chunk0, n, final_idx, 0});
    return chunk0;
  }

  // One segment cut into 128-row tiles; tile j starts from stateA[a] plus
  // the prefix slot of its first chunk (none for j = 0).
  void add_segment_tiles(int64_t start, int64_t len, int stateA, int chunk0) {
    for (int64_t r = 0; r < len; r += kTileRows) {
      const int j = static_cast<int>(r / kTileRows);
      TileDesc t{};
      t.row0 = static_cast<int32_t>(start + r);
      t.nrows = static_cast<int32_t>(std::min<int64_t>(kTileRows, len - r));
      t.stateA = stateA;
      t.stateB = j == 0 ? -1 : chunk0 + 2 * j;
      t.bound0 = static_cast<int32_t>(bounds.size());
      t.nbound = 1;
      bounds.push_back(0);
      tiles.push_back(t);
    }
  }

  // Branches: short ones (<= 128 rows) are packed greedily with adjacent,
  // contiguous branches of the same parent; longer ones are chunked and
  // scanned like views and start every tile from parent + prefix.
  void add_branches(const int32_t* cu, int32_t B, const int32_t* parent) {
    int open = -1;   // index of the short-branch tile being filled
    for (int32_t b = 0; b < B; ++b) {
      const int64_t start = cu[b], len = cu[b + 1] - cu[b];
      if (len == 0) continue;
      if (len > kTileRows) {
        open = -1;
        const int chunk0 = add_chunks(start, len, -1);
        add_segment_tiles(start, len, parent[b], chunk0);
        continue;
      }
      if (open >= 0) {
        TileDesc& t = tiles[open];
        if (t.stateA == parent[b] && t.row0 + t.nrows == start && t.nrows + len <= kTileRows) {
          bounds.push_back(static_cast<uint8_t>(t.nrows));
          t.nbound += 1;
          t.nrows += static_cast<int32_t>(len);
          continue;
        }
      }
      TileDesc t{};
      t.row0 = static_cast<int32_t>(start);
      t.nrows = static_cast<int32_t>(len);
      t.stateA = parent[b];
      t.stateB = -1;
      t.bound0 = static_cast<int32_t>(bounds.size());
      t.nbound = 1;
      bounds.push_back(0);
      open = static_cast<int>(tiles.size());
      tiles.push_back(t);
    }
  }
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Workspace {
  size_t off_tiles = 0, off_chunks = 0, off_scan = 0, off_bounds = 0, desc_bytes = 0;
  size_t off_states = 0, off_parts = 0, total = 0;
};

Workspace layout(const Plan& p, int H, int64_t T, bool split) {
  Workspace w;
  size_t o = 0;
  w.off_tiles = o;  o = align256(o + p.tiles.size() * sizeof(TileDesc));
  w.off_chunks = o; o = align256(o + p.chunks.size() * sizeof(ChunkDesc));
  w.off_scan = o;   o = align256(o + p.scan.size() * sizeof(ScanDesc));
  w.off_bounds = o; o = align256(o + p.bounds.size());
  w.desc_bytes = o;
  w.off_states = o; o = align256(o + p.chunks.size() * static_cast<size_t>(H) * kStateFloats * sizeof(float));
  w.off_parts = o;
  if (split) o = align256(o + 6 * static_cast<size_t>(T) * H * kHeadDim * 2);
  w.total = o;
  return w;
}

// 3-D view (d, token, head) of a [T][H][64] bf16 array; box = {64, rows, heads}.
span_la_status encode_map(CUtensorMap* map, const void* base, int64_t T, int H, int box_rows,
                          int box_heads) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(T),
                              static_cast<cuuint64_t>(H)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(H) * kHeadDim * 2, kHeadDim * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), static_cast<cuuint32_t>(box_rows),
                             static_cast<cuuint32_t>(box_heads)};
  const cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPAN_LA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return SPAN_LA_OK;
}

// Common tail of both entry points: workspace, descriptor upload, launches.
span_la_status run_plan(const Plan& plan, const void* q, const void* k, const void* v,
                        const span_la_dims& dims, const float* stateA, float* final_out,
                        void* out, cudaStream_t stream, DeviceState* dev) {
  const int H = dims.num_heads;
  const int64_t T = dims.total_rows;
  const bool split = dims.dtype == SPAN_LA_F32;
  if (plan.tiles.empty() && plan.scan.empty()) return SPAN_LA_OK;

  const Workspace w = layout(plan, H, T, split);
  std::vector<uint8_t> host(w.desc_bytes, 0);
  if (!plan.tiles.empty()) std::memcpy(host.data() + w.off_tiles, plan.tiles.data(), plan.tiles.size() * sizeof(TileDesc));
  if (!plan.chunks.empty()) std::memcpy(host.data() + w.off_chunks, plan.chunks.data(), plan.chunks.size() * sizeof(ChunkDesc));
  if (!plan.scan.empty()) std::memcpy(host.data() + w.off_scan, plan.scan.data(), plan.scan.size() * sizeof(ScanDesc));
  if (!plan.bounds.empty()) std::memcpy(host.data() + w.off_bounds, plan.bounds.data(), plan.bounds.size());

  uint8_t* ws = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&ws), w.total, stream);
  if (e != cudaSuccess) return fail(SPAN_LA_ERR_NOMEM, "cudaMallocAsync(%zu): %s", w.total, cudaGetErrorString(e));
  span_la_status st = SPAN_LA_OK;
  do {
    e = cudaMemcpyAsync(ws, host.data(), w.desc_bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) { st = cuda_fail(e, "cudaMemcpyAsync(descriptors)"); break; }

    // bf16 operand arrays the kernels read through TMA: the inputs themselves,
    // or, for fp32 inputs, their bf16 high / low parts made by the split kernel.
    const void* parts[3][2] = {{q, nullptr}, {k, nullptr}, {v, nullptr}};
    if (split) {
      const size_t part_bytes = static_cast<size_t>(T) * H * kHeadDim * 2;
      for (int t = 0; t < 3; ++t)
        for (int p = 0; p < 2; ++p) parts[t][p] = ws + w.off_parts + (2 * t + p) * part_bytes;
      e = launch_split_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                           static_cast<const float*>(v), T * H * kHeadDim, ws + w.off_parts, stream);
      if (e != cudaSuccess) { st = cuda_fail(e, "split kernel launch"); break; }
    }
    DeviceOperands tile_ops{}, chunk_ops{};
    const bool need_maps = !plan.tiles.empty() || !plan.chunks.empty();   // implies T > 0
    for (int t = 0; t < 3 && st == SPAN_LA_OK && need_maps; ++t) {
      for (int p = 0; p < (split ? 2 : 1) && st == SPAN_LA_OK; ++p) {
        CUtensorMap* tm = t == 0 ? &tile_ops.q[p] : t == 1 ? &tile_ops.k[p] : &tile_ops.v[p];
        CUtensorMap* cm = t == 0 ? &chunk_ops.q[p] : t == 1 ? &chunk_ops.k[p] : &chunk_ops.v[p];
        st = encode_map(tm, parts[t][p], T, H, kTileBoxRows, 1);
        if (st == SPAN_LA_OK && t > 0) st = encode_map(cm, parts[t][p], T, H, kChunkBoxRows, kChunkBoxHeads);
      }
    }
    if (st != SPAN_LA_OK) break;

    float* states = reinterpret_cast<float*>(ws + w.off_states);
    e = launch_chunk_state(split, chunk_ops.k, chunk_ops.v, reinterpret_cast<const ChunkDesc*>(ws + w.off_chunks),
                           static_cast<int>(plan.chunks.size()), H, states, dev->err, stream);
    if (e != cudaSuccess) { st = cuda_fail(e, "chunk-state launch"); break; }
    e = launch_scan(reinterpret_cast<const ScanDesc*>(ws + w.off_scan), static_cast<int>(plan.scan.size()), H,
                    states, final_out, stream);
    if (e != cudaSuccess) { st = cuda_fail(e, "scan launch"); break; }
    e = launch_tile_output(split, tile_ops.q, tile_ops.k, tile_ops.v,
                           reinterpret_cast<const TileDesc*>(ws + w.off_tiles), static_cast<int>(plan.tiles.size()),
                           ws + w.off_bounds, stateA, states, out, H, dev->err, stream);
    if (e != cudaSuccess) { st = cuda_fail(e, "tile-output launch"); break; }
  } while (false);
  cudaError_t ef = cudaFreeAsync(ws, stream);
  if (st == SPAN_LA_OK && ef != cudaSuccess) st = cuda_fail(ef, "cudaFreeAsync");
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

  Plan plan;
  for (int32_t s = 0; s < num_views; ++s) {
    const int64_t start = view_cu_seqlens[s], len = view_cu_seqlens[s + 1] - view_cu_seqlens[s];
    const int chunk0 = plan.add_chunks(start, len, s);
    plan.add_segment_tiles(start, len, -1, chunk0);
  }
  if (num_branches > 0) plan.add_branches(branch_cu_seqlens, num_branches, branch_parent);
  return run_plan(plan, q, k, v, dims, view_state_out, view_state_out, out, stream, dev);
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

  Plan plan;
  plan.add_branches(branch_cu_seqlens, num_branches, branch_parent);
  return run_plan(plan, q, k, v, dims, cached_state, nullptr, out, stream, dev);
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
  if (word != 0) {
    cudaMemset(dev->err, 0, sizeof(unsigned));
    return fail(SPAN_LA_ERR_TIMEOUT, "a bounded device wait ran out (error word 0x%x)", word);
  }
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

int32_t span_la_version(void) { return 100; }

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
