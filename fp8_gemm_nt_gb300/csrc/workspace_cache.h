// Per-stream device workspaces: the cache policy, written against a small API so that the host
// logic can be checked without a GPU (tests/workspace_cache_check.cpp runs it on fake calls).
//
// One workspace per stream. Rules:
//   * Nothing here synchronises the device or a stream. Blocks are allocated and freed in
//     stream order (cudaMallocAsync / cudaFreeAsync on the requesting stream), so a call that
//     needs a new or larger block costs an allocation, never a wait.
//   * A reserved workspace (dg_reserve_workspace) is allocated up front and kept until the
//     caller releases it: calls on its stream that fit it allocate, free and synchronise
//     nothing. It grows (in stream order) if a call needs more than was reserved.
//   * At most kMaxFreeable workspaces that are neither reserved nor referenced by a graph are
//     kept. A request from a further stream evicts the least recently used one: the requesting
//     stream waits (on the device) for that workspace's last use, an event recorded after its
//     last launch, and frees it in its own order. The evicted stream may already be destroyed:
//     only the event is used.
//   * A workspace used while its stream is being captured into a CUDA graph is referenced by
//     that graph, whose replays may come at any later time. It is marked captured and never
//     freed. Growing it moves the old block to `retained`, which also lives until exit.
//   * While the requesting stream is being captured nothing is freed or evicted, and a block
//     allocated then comes from the synchronous allocator (a stream-ordered allocation would
//     become a node of the graph); it is zeroed by a memset that becomes part of the graph.
// The caller serialises calls (one lock) and keeps that lock until the kernels that use the
// returned block are enqueued and release() has recorded the last-use event, so an eviction
// in another host thread always orders its free after those kernels.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <type_traits>
#include <vector>

namespace dg {

template <class Stream, class Event>
struct Workspace {
  Stream stream{};
  void* ptr = nullptr;
  size_t bytes = 0;
  bool captured = false;   // a graph refers to it: never freed
  bool reserved = false;   // kept until dg_release_workspace
  bool async = false;      // allocated in stream order (freeable in stream order)
  bool has_event = false;  // `last_use` holds the point after its last launch
  Event last_use{};
  uint64_t tick = 0;       // recency, for eviction
};

template <class Stream, class Event>
struct WorkspaceCache {
  std::vector<Workspace<Stream, Event>> live;
  std::vector<Workspace<Stream, Event>> retained;   // blocks a captured graph may still use
  uint64_t clock = 0;
};

// Api: using Stream, Event; each call returns 0 on success, else an error code:
//   is_capturing(Stream, bool*), malloc(void**, size_t) (synchronous allocator, for captures),
//   malloc_async(void**, size_t, Stream), free_async(void*, Stream), memset_async(void*, size_t,
//   Stream), event_create(Event*), event_destroy(Event), event_record(Event, Stream),
//   stream_wait_event(Stream, Event).

namespace detail {

template <class Api, class WS>
int drop_event(WS& w) {
  if (w.has_event) {
    w.has_event = false;
    if (int e = Api::event_destroy(w.last_use)) return e;
  }
  return 0;
}

// Frees w's block in the order of `stream` (after w's last use, which may be on another stream).
template <class Api, class WS>
int free_in_order(WS& w, typename Api::Stream stream) {
  if (w.ptr && w.async) {
    if (w.has_event && w.stream != stream)
      if (int e = Api::stream_wait_event(stream, w.last_use)) return e;
    if (int e = Api::free_async(w.ptr, stream)) return e;
  }
  w.ptr = nullptr;
  w.bytes = 0;
  return drop_event<Api>(w);
}

// The entry of `stream`, created if missing. A new entry beyond the freeable cap evicts the
// least recently used freeable one (not while capturing).
template <class Api, size_t kMaxFreeable, class Cache>
int entry(Cache& cache, typename Api::Stream stream, bool capturing, size_t* index) {
  using WS = typename std::decay<decltype(cache.live[0])>::type;
  for (size_t i = 0; i < cache.live.size(); ++i)
    if (cache.live[i].stream == stream) {
      *index = i;
      return 0;
    }
  auto freeable = [](const WS& x) { return !x.captured && !x.reserved; };
  if (!capturing &&
      static_cast<size_t>(std::count_if(cache.live.begin(), cache.live.end(), freeable)) >= kMaxFreeable) {
    size_t victim = cache.live.size();
    for (size_t i = 0; i < cache.live.size(); ++i)
      if (freeable(cache.live[i]) && (victim == cache.live.size() || cache.live[i].tick < cache.live[victim].tick))
        victim = i;
    if (victim < cache.live.size()) {
      if (int e = free_in_order<Api>(cache.live[victim], stream)) return e;
      cache.live.erase(cache.live.begin() + static_cast<std::ptrdiff_t>(victim));
    }
  }
  WS w;
  w.stream = stream;
  cache.live.push_back(w);
  *index = cache.live.size() - 1;
  return 0;
}

// Makes cache.live[i] at least `bytes` (a new block zero-filled); `slack` over-allocates.
template <class Api, class Cache>
int grow(Cache& cache, size_t i, typename Api::Stream stream, size_t bytes, bool capturing, bool slack) {
  auto& w = cache.live[i];
  if (w.bytes >= bytes) return 0;
  if (w.ptr) {
    if (w.captured || capturing) {
      cache.retained.push_back(w);   // a graph may use it (or is being recorded with it)
      w.ptr = nullptr;
      w.bytes = 0;
      w.has_event = false;           // the event (if any) goes with the retained entry
    } else if (int e = free_in_order<Api>(w, stream)) {
      return e;
    }
  }
  const size_t alloc = slack ? bytes + bytes / 2 : bytes;
  if (capturing) {
    if (int e = Api::malloc(&w.ptr, alloc)) {
      w.ptr = nullptr;
      return e;
    }
    w.async = false;
  } else {
    if (int e = Api::malloc_async(&w.ptr, alloc, stream)) {
      w.ptr = nullptr;
      return e;
    }
    w.async = true;
  }
  w.bytes = alloc;
  w.captured = false;
  return Api::memset_async(w.ptr, alloc, stream);
}

}  // namespace detail

// The workspace of `stream`, at least `bytes`, zero-filled when newly allocated: *out and its
// entry index. Call release() once the kernels that use it are enqueued.
template <class Api, size_t kMaxFreeable, class Cache>
int acquire(Cache& cache, typename Api::Stream stream, size_t bytes, void** out, size_t* index) {
  bool capturing = false;
  if (int e = Api::is_capturing(stream, &capturing)) return e;
  size_t i = 0;
  if (int e = detail::entry<Api, kMaxFreeable>(cache, stream, capturing, &i)) return e;
  if (int e = detail::grow<Api>(cache, i, stream, bytes, capturing, true)) return e;
  auto& w = cache.live[i];
  if (capturing) w.captured = true;
  w.tick = ++cache.clock;
  *out = w.ptr;
  *index = i;
  return 0;
}

// After the launches that use entry `index` (returned by acquire) are enqueued on `stream`:
// a freeable workspace records the point after them, for a later eviction from another stream.
template <class Api, class Cache>
int release(Cache& cache, size_t index, typename Api::Stream stream) {
  auto& w = cache.live[index];
  if (w.captured || w.reserved) return 0;
  bool capturing = false;
  if (int e = Api::is_capturing(stream, &capturing)) return e;
  if (capturing) return 0;
  if (!w.has_event) {
    if (int e = Api::event_create(&w.last_use)) return e;
    w.has_event = true;
  }
  return Api::event_record(w.last_use, stream);
}

// dg_reserve_workspace: the workspace of `stream` becomes at least `bytes` (allocated now, in
// stream order) and is kept until reserve_release(). Refused (returns -1) while the stream is
// being captured.
template <class Api, size_t kMaxFreeable, class Cache>
int reserve(Cache& cache, typename Api::Stream stream, size_t bytes) {
  bool capturing = false;
  if (int e = Api::is_capturing(stream, &capturing)) return e;
  if (capturing) return -1;
  size_t i = 0;
  if (int e = detail::entry<Api, kMaxFreeable>(cache, stream, false, &i)) return e;
  if (int e = detail::grow<Api>(cache, i, stream, bytes, false, false)) return e;
  auto& w = cache.live[i];
  w.reserved = true;
  w.tick = ++cache.clock;
  return detail::drop_event<Api>(w);
}

// dg_release_workspace: frees the workspace of `stream` in that stream's order (a block a
// graph refers to is kept until exit instead). Refused (returns -1) while capturing.
template <class Api, class Cache>
int reserve_release(Cache& cache, typename Api::Stream stream) {
  bool capturing = false;
  if (int e = Api::is_capturing(stream, &capturing)) return e;
  if (capturing) return -1;
  for (size_t i = 0; i < cache.live.size(); ++i) {
    auto& w = cache.live[i];
    if (w.stream != stream) continue;
    if (w.captured) {
      cache.retained.push_back(w);
    } else if (int e = detail::free_in_order<Api>(w, stream)) {
      return e;
    }
    cache.live.erase(cache.live.begin() + static_cast<std::ptrdiff_t>(i));
    return 0;
  }
  return 0;
}

// Bytes of the workspace `stream` has (0: none).
template <class Cache, class Stream>
size_t workspace_bytes(const Cache& cache, Stream stream) {
  for (const auto& w : cache.live)
    if (w.stream == stream) return w.bytes;
  return 0;
}

}  // namespace dg
