// View-state cache of libspanla: view final states kept in device memory
// under caller keys, so that the branches of a long request (or its shards)
// start from the cached state instead of recomputing the view.
//
// "Serving 0.88M TPS from Two RTXs and Mac Minis", section "Long Requests":
// shards of a long request reuse the view's cached state; without the cache
// the same work took 3.4x as long.
//
// The cache is host bookkeeping (key -> slot, a use clock per slot for the
// least-recently-used eviction) over one device array of `capacity` states.
// Puts copy states in with cudaMemcpyAsync on the caller's stream; branch
// calls map their parent keys to slots and run span_la_branches_from_state
// over the device array.  Each slot carries CUDA events for its last write
// (a put) and for its last read on each stream (branch calls), so that a
// branch call waits for the put of its state and a put that reuses a slot
// waits for every read of the state it replaces, whichever streams they ran on.
#include <algorithm>
#include <cstdio>
#include <cstdarg>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include <cuda_runtime.h>

#include "spanla.h"
#include "spanla_internal.h"

struct span_la_view_cache {
  struct Reader {
    cudaStream_t stream;
    cudaEvent_t done;     // recorded after that stream's last branch call on the slot
  };
  int device = 0;
  int heads = 0;
  int capacity = 0;
  float* pool = nullptr;                      // [capacity][heads][64][64]
  std::unordered_map<uint64_t, int32_t> slot_of;
  std::vector<uint64_t> key_of;               // per slot (valid when used[slot])
  std::vector<char> used;
  std::vector<uint64_t> last_use;
  std::vector<cudaEvent_t> written;           // per slot: after its last put
  std::vector<char> has_written;
  std::vector<std::vector<Reader>> readers;   // per slot, since its last put
  std::vector<cudaEvent_t> spare_events;
  uint64_t clock = 0;
  int64_t hits = 0, misses = 0, evictions = 0, puts = 0;
  mutable std::mutex mu;
};

namespace {

constexpr size_t kStateBytesPerHead = static_cast<size_t>(spanla::kStateFloats) * sizeof(float);

span_la_status cache_fail(span_la_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  spanla::set_last_error_detail(buf);   // what span_la_last_error_detail() returns
  return s;
}

// A slot for a new key: a free one, else the least recently used slot whose
// key is not in `keep`.  -1 if none.
int32_t take_slot(span_la_view_cache* c, const std::unordered_set<uint64_t>& keep) {
  for (int32_t s = 0; s < c->capacity; ++s)
    if (!c->used[s]) return s;
  int32_t victim = -1;
  for (int32_t s = 0; s < c->capacity; ++s) {
    if (keep.count(c->key_of[s])) continue;
    if (victim < 0 || c->last_use[s] < c->last_use[victim]) victim = s;
  }
  if (victim >= 0) {
    c->slot_of.erase(c->key_of[victim]);
    c->used[victim] = 0;
    c->evictions += 1;
  }
  return victim;
}

cudaError_t new_event(span_la_view_cache* c, cudaEvent_t* ev) {
  if (!c->spare_events.empty()) {
    *ev = c->spare_events.back();
    c->spare_events.pop_back();
    return cudaSuccess;
  }
  return cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
}

// Make `stream` wait until every earlier read and write of `slot` is done.
cudaError_t order_before_write(span_la_view_cache* c, int32_t slot, cudaStream_t stream) {
  for (const auto& r : c->readers[slot]) {
    cudaError_t e = cudaStreamWaitEvent(stream, r.done, 0);
    if (e != cudaSuccess) return e;
    c->spare_events.push_back(r.done);
  }
  c->readers[slot].clear();
  if (c->has_written[slot]) return cudaStreamWaitEvent(stream, c->written[slot], 0);
  return cudaSuccess;
}

// Record on `stream` that it has enqueued a read of `slot`.
cudaError_t note_read(span_la_view_cache* c, int32_t slot, cudaStream_t stream) {
  for (auto& r : c->readers[slot])
    if (r.stream == stream) return cudaEventRecord(r.done, stream);
  span_la_view_cache::Reader r{stream, nullptr};
  cudaError_t e = new_event(c, &r.done);
  if (e == cudaSuccess) e = cudaEventRecord(r.done, stream);
  if (e == cudaSuccess) c->readers[slot].push_back(r);
  return e;
}

void release_events(span_la_view_cache* c) {
  for (int32_t s = 0; s < static_cast<int32_t>(c->written.size()); ++s) {
    if (c->written[s] != nullptr) cudaEventDestroy(c->written[s]);
    for (const auto& r : c->readers[s]) cudaEventDestroy(r.done);
  }
  for (cudaEvent_t e : c->spare_events) cudaEventDestroy(e);
  c->written.clear();
  c->readers.clear();
  c->spare_events.clear();
}

// The cache's cross-stream events are host-side state of each call, so its
// calls are not recorded into CUDA graphs.
// Calls run on the device the cache was created on.
span_la_status check_device(const span_la_view_cache* c) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cache_fail(SPAN_LA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev != c->device)
    return cache_fail(SPAN_LA_ERR_INVALID, "the current device is %d; the cache lives on device %d", dev,
                      c->device);
  return SPAN_LA_OK;
}

span_la_status refuse_capture(cudaStream_t stream) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cache_fail(SPAN_LA_ERR_CUDA, "cudaStreamIsCapturing: %s", cudaGetErrorString(e));
  if (cap != cudaStreamCaptureStatusNone)
    return cache_fail(SPAN_LA_ERR_UNSUPPORTED, "view-state cache calls cannot be captured into a CUDA graph");
  return SPAN_LA_OK;
}

}  // namespace

extern "C" {

span_la_status span_la_cache_create(int32_t num_heads, int32_t capacity, span_la_view_cache** cache) {
  if (cache == nullptr) return cache_fail(SPAN_LA_ERR_INVALID, "cache is NULL");
  *cache = nullptr;
  if (num_heads < 1) return cache_fail(SPAN_LA_ERR_INVALID, "num_heads %d < 1", num_heads);
  if (capacity < 1) return cache_fail(SPAN_LA_ERR_INVALID, "capacity %d < 1", capacity);
  span_la_view_cache* c = new span_la_view_cache();
  c->heads = num_heads;
  c->capacity = capacity;
  cudaError_t e = cudaGetDevice(&c->device);
  if (e != cudaSuccess) {
    delete c;
    return cache_fail(SPAN_LA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  }
  const size_t bytes = static_cast<size_t>(capacity) * num_heads * kStateBytesPerHead;
  e = cudaMalloc(reinterpret_cast<void**>(&c->pool), bytes);
  if (e != cudaSuccess) {
    delete c;
    return cache_fail(SPAN_LA_ERR_NOMEM, "cudaMalloc(%zu bytes of view states): %s", bytes,
                      cudaGetErrorString(e));
  }
  c->key_of.assign(capacity, 0);
  c->used.assign(capacity, 0);
  c->last_use.assign(capacity, 0);
  c->written.assign(capacity, nullptr);
  c->has_written.assign(capacity, 0);
  c->readers.resize(capacity);
  for (int32_t s = 0; s < capacity && e == cudaSuccess; ++s)
    e = cudaEventCreateWithFlags(&c->written[s], cudaEventDisableTiming);
  if (e != cudaSuccess) {
    release_events(c);
    cudaFree(c->pool);
    delete c;
    return cache_fail(SPAN_LA_ERR_CUDA, "cudaEventCreate: %s", cudaGetErrorString(e));
  }
  *cache = c;
  return SPAN_LA_OK;
}

span_la_status span_la_cache_destroy(span_la_view_cache* cache) {
  if (cache == nullptr) return SPAN_LA_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(cache->device);
  cudaError_t e = cudaDeviceSynchronize();
  release_events(cache);
  if (e == cudaSuccess) e = cudaFree(cache->pool);
  cudaSetDevice(prev);
  delete cache;
  if (e != cudaSuccess) return cache_fail(SPAN_LA_ERR_CUDA, "cache destroy: %s", cudaGetErrorString(e));
  return SPAN_LA_OK;
}

span_la_status span_la_cache_put(span_la_view_cache* cache, const uint64_t* keys, int32_t n,
                                 const float* states, cudaStream_t stream) {
  if (cache == nullptr) return cache_fail(SPAN_LA_ERR_INVALID, "cache is NULL");
  if (n < 1 || n > cache->capacity)
    return cache_fail(SPAN_LA_ERR_INVALID, "n = %d not in [1, capacity %d]", n, cache->capacity);
  if (keys == nullptr || states == nullptr) return cache_fail(SPAN_LA_ERR_INVALID, "keys or states is NULL");
  if ((reinterpret_cast<uintptr_t>(states) & 15u) != 0)
    return cache_fail(SPAN_LA_ERR_INVALID, "states must be 16-byte aligned");
  std::unordered_set<uint64_t> keep(keys, keys + n);
  if (static_cast<int32_t>(keep.size()) != n) return cache_fail(SPAN_LA_ERR_INVALID, "keys are not distinct");
  span_la_status cst = check_device(cache);
  if (cst == SPAN_LA_OK) cst = refuse_capture(stream);
  if (cst != SPAN_LA_OK) return cst;
  std::lock_guard<std::mutex> lock(cache->mu);
  const size_t state_bytes = static_cast<size_t>(cache->heads) * kStateBytesPerHead;
  for (int32_t i = 0; i < n; ++i) {
    auto it = cache->slot_of.find(keys[i]);
    int32_t slot = it != cache->slot_of.end() ? it->second : take_slot(cache, keep);
    if (slot < 0) return cache_fail(SPAN_LA_ERR_INVALID, "no slot left for key %d of the put", i);
    cudaError_t e = order_before_write(cache, slot, stream);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(cache->pool + static_cast<size_t>(slot) * cache->heads * spanla::kStateFloats,
                          states + static_cast<size_t>(i) * cache->heads * spanla::kStateFloats,
                          state_bytes, cudaMemcpyDeviceToDevice, stream);
    if (e == cudaSuccess) e = cudaEventRecord(cache->written[slot], stream);
    if (e != cudaSuccess) {
      // The slot's contents are unknown now: drop its key.
      if (cache->used[slot]) cache->slot_of.erase(cache->key_of[slot]);
      cache->used[slot] = 0;
      return cache_fail(SPAN_LA_ERR_CUDA, "view state put: %s", cudaGetErrorString(e));
    }
    cache->has_written[slot] = 1;
    cache->slot_of[keys[i]] = slot;
    cache->key_of[slot] = keys[i];
    cache->used[slot] = 1;
    cache->last_use[slot] = ++cache->clock;
    cache->puts += 1;
  }
  return SPAN_LA_OK;
}

span_la_status span_la_cache_contains(span_la_view_cache* cache, const uint64_t* keys, int32_t n,
                                      int32_t* present) {
  if (cache == nullptr) return cache_fail(SPAN_LA_ERR_INVALID, "cache is NULL");
  if (n < 0 || (n > 0 && (keys == nullptr || present == nullptr)))
    return cache_fail(SPAN_LA_ERR_INVALID, "bad key arrays");
  std::lock_guard<std::mutex> lock(cache->mu);
  for (int32_t i = 0; i < n; ++i) {
    auto it = cache->slot_of.find(keys[i]);
    present[i] = it != cache->slot_of.end();
    if (present[i]) {
      cache->last_use[it->second] = ++cache->clock;
      cache->hits += 1;
    } else {
      cache->misses += 1;
    }
  }
  return SPAN_LA_OK;
}

span_la_status span_la_cache_branches(span_la_view_cache* cache, const uint64_t* parent_keys,
                                      const void* q, const void* k, const void* v, span_la_dims dims,
                                      const int32_t* branch_cu_seqlens, int32_t num_branches, void* out,
                                      cudaStream_t stream) {
  if (cache == nullptr) return cache_fail(SPAN_LA_ERR_INVALID, "cache is NULL");
  if (dims.num_heads != cache->heads)
    return cache_fail(SPAN_LA_ERR_INVALID, "num_heads %d differs from the cache's %d", dims.num_heads,
                      cache->heads);
  if (num_branches < 0 || (num_branches > 0 && parent_keys == nullptr))
    return cache_fail(SPAN_LA_ERR_INVALID, "bad parent key array");
  span_la_status cst = check_device(cache);
  if (cst == SPAN_LA_OK) cst = refuse_capture(stream);
  if (cst != SPAN_LA_OK) return cst;
  std::vector<int32_t> slots(num_branches);
  {
    std::lock_guard<std::mutex> lock(cache->mu);
    for (int32_t b = 0; b < num_branches; ++b) {
      auto it = cache->slot_of.find(parent_keys[b]);
      if (it == cache->slot_of.end()) {
        cache->misses += 1;
        return cache_fail(SPAN_LA_ERR_INVALID, "parent key of branch %d is not cached", b);
      }
      slots[b] = it->second;
    }
    // Only a call that will run counts as a use of its entries.
    for (int32_t b = 0; b < num_branches; ++b) {
      cache->last_use[slots[b]] = ++cache->clock;
      cache->hits += 1;
    }
    // Wait for the puts of these states (a no-op on the put's own stream),
    // enqueue, then record the reads, all under the lock so that no put of
    // another thread can reuse these slots in between.
    std::vector<int32_t> distinct(slots);
    std::sort(distinct.begin(), distinct.end());
    distinct.erase(std::unique(distinct.begin(), distinct.end()), distinct.end());
    for (int32_t slot : distinct) {
      cudaError_t e = cudaStreamWaitEvent(stream, cache->written[slot], 0);
      if (e != cudaSuccess) return cache_fail(SPAN_LA_ERR_CUDA, "cudaStreamWaitEvent: %s", cudaGetErrorString(e));
    }
    span_la_status st = span_la_branches_from_state(cache->pool, cache->capacity, q, k, v, dims,
                                                    branch_cu_seqlens, num_branches, slots.data(), out,
                                                    stream);
    if (st != SPAN_LA_OK) return st;
    for (int32_t slot : distinct) {
      cudaError_t e = note_read(cache, slot, stream);
      if (e != cudaSuccess) return cache_fail(SPAN_LA_ERR_CUDA, "cudaEventRecord: %s", cudaGetErrorString(e));
    }
    return SPAN_LA_OK;
  }
}

span_la_status span_la_cache_stats(const span_la_view_cache* cache, int64_t* stats) {
  if (cache == nullptr || stats == nullptr) return cache_fail(SPAN_LA_ERR_INVALID, "cache or stats is NULL");
  std::lock_guard<std::mutex> lock(cache->mu);
  stats[0] = static_cast<int64_t>(cache->slot_of.size());
  stats[1] = cache->capacity;
  stats[2] = cache->hits;
  stats[3] = cache->misses;
  stats[4] = cache->evictions;
  stats[5] = cache->puts;
  return SPAN_LA_OK;
}

}  // extern "C"
