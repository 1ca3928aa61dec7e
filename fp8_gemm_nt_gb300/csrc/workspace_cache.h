// Per-stream device workspaces: the cache policy, written against a small API so that the host
// logic can be checked without a GPU (tests/workspace_cache_check.cpp runs it on fake calls).
//
// One workspace per stream, grown on demand. Rules:
//   * At most kMaxFreeable workspaces that no graph refers to are kept. A request from a
//     further stream first waits for the device, so that every workspace is idle, and then
//     frees them. Streams come and go, and a workspace is not tied to its stream's lifetime.
//   * A workspace used while its stream is being captured into a CUDA graph is referenced by
//     that graph, whose replays may come at any later time. It is marked captured and never
//     freed. Growing it moves the old block to `retained`, which also lives until exit.
//   * While the requesting stream is being captured nothing is synchronised or freed (neither
//     is allowed during a capture). A block allocated then is zeroed by a memset that becomes
//     part of the graph.
// The caller serialises calls (one lock) and keeps that lock until the kernels that use the
// returned block are enqueued, so a later synchronisation before a free waits for them.
#pragma once

#include <algorithm>
#include <cstddef>
#include <vector>

namespace dg {

template <class Stream>
struct Workspace {
  Stream stream{};
  void* ptr = nullptr;
  size_t bytes = 0;
  bool captured = false;
};

template <class Stream>
struct WorkspaceCache {
  std::vector<Workspace<Stream>> live;
  std::vector<Workspace<Stream>> retained;   // blocks a captured graph may still use
};

// Api: using Stream; static int is_capturing(Stream, bool*), device_synchronize(),
// stream_synchronize(Stream), malloc(void**, size_t), free(void*),
// memset_async(void*, size_t, Stream): each returns 0 on success, else an error code.
// acquire() returns 0 and sets *out (at least `bytes`, zero-filled when newly allocated), or
// the first error code.
template <class Api, size_t kMaxFreeable>
int acquire(WorkspaceCache<typename Api::Stream>& cache, typename Api::Stream stream, size_t bytes, void** out) {
  using WS = Workspace<typename Api::Stream>;
  bool capturing = false;
  if (int e = Api::is_capturing(stream, &capturing)) return e;
  WS* w = nullptr;
  for (auto& x : cache.live)
    if (x.stream == stream) w = &x;
  if (!w) {
    const auto freeable = static_cast<size_t>(
        std::count_if(cache.live.begin(), cache.live.end(), [](const WS& x) { return !x.captured; }));
    if (freeable >= kMaxFreeable && !capturing) {
      if (int e = Api::device_synchronize()) return e;
      for (auto& x : cache.live)
        if (!x.captured && x.ptr)
          if (int e = Api::free(x.ptr)) return e;
      cache.live.erase(std::remove_if(cache.live.begin(), cache.live.end(), [](const WS& x) { return !x.captured; }),
                       cache.live.end());
    }
    cache.live.push_back(WS{stream, nullptr, 0, false});
    w = &cache.live.back();
  }
  if (w->bytes < bytes) {
    if (w->ptr) {
      if (w->captured || capturing) {
        cache.retained.push_back(*w);
      } else {
        if (int e = Api::stream_synchronize(stream)) return e;
        if (int e = Api::free(w->ptr)) return e;
      }
      w->ptr = nullptr;
      w->bytes = 0;
      w->captured = false;
    }
    const size_t alloc = bytes + bytes / 2;
    if (int e = Api::malloc(&w->ptr, alloc)) {
      w->ptr = nullptr;
      return e;
    }
    w->bytes = alloc;
    if (int e = Api::memset_async(w->ptr, alloc, stream)) return e;
  }
  if (capturing) w->captured = true;
  *out = w->ptr;
  return 0;
}

}  // namespace dg
