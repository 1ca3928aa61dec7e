// Host-only check of the per-stream workspace cache policy (workspace_cache.h) on fake CUDA
// calls. The fakes assert the two safety rules: no block that a captured graph refers to is
// ever freed, and nothing is synchronised while the requesting stream is being captured.
// Prints "ok" and exits 0 when every scenario holds.
#include <cassert>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <set>

#include "workspace_cache.h"

namespace {

struct FakeStream;
using Stream = FakeStream*;

std::set<void*> live;         // blocks allocated and not freed
std::set<void*> graph_refs;   // blocks a captured launch refers to
std::set<Stream> capturing;
int device_syncs = 0, frees = 0, memsets = 0;

#define CHECK(cond)                                                     \
  do {                                                                  \
    if (!(cond)) {                                                      \
      std::fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
      std::exit(1);                                                     \
    }                                                                   \
  } while (0)

struct FakeApi {
  using Stream = ::Stream;
  static int is_capturing(Stream s, bool* c) {
    *c = capturing.count(s) != 0;
    return 0;
  }
  static int device_synchronize() {
    CHECK(capturing.empty());
    ++device_syncs;
    return 0;
  }
  static int stream_synchronize(Stream s) {
    CHECK(!capturing.count(s));
    return 0;
  }
  static int malloc(void** p, size_t n) {
    *p = std::malloc(n);
    live.insert(*p);
    return 0;
  }
  static int free(void* p) {
    CHECK(live.count(p));
    CHECK(!graph_refs.count(p));
    live.erase(p);
    std::free(p);
    ++frees;
    return 0;
  }
  static int memset_async(void*, size_t, Stream) {
    ++memsets;
    return 0;
  }
};

constexpr size_t kCap = 16;

Stream S(int i) { return reinterpret_cast<Stream>(static_cast<uintptr_t>(0x1000 + 16 * i)); }

void* call(dg::WorkspaceCache<Stream>& c, int s, size_t bytes) {
  void* p = nullptr;
  CHECK((dg::acquire<FakeApi, kCap>(c, S(s), bytes, &p) == 0));
  CHECK(p && live.count(p));
  if (capturing.count(S(s))) graph_refs.insert(p);   // the captured launch refers to it
  return p;
}

size_t freeable(const dg::WorkspaceCache<Stream>& c) {
  size_t n = 0;
  for (const auto& w : c.live) n += !w.captured;
  return n;
}

}  // namespace

int main() {
  dg::WorkspaceCache<Stream> c;
  // streams come and go: at most kCap freeable entries, memory stays bounded
  for (int r = 0; r < 3; ++r)
    for (int s = 0; s < 40; ++s) {
      call(c, s, 1000);
      CHECK(freeable(c) <= kCap);
    }
  CHECK(device_syncs > 0 && live.size() <= kCap);
  // the same stream reuses its block; a larger request on an uncaptured stream frees the old one
  void* u0 = call(c, 600, 100);
  CHECK(call(c, 600, 100) == u0);
  const int f0 = frees;
  void* u1 = call(c, 600, 10000);
  CHECK(u1 != u0 && !live.count(u0) && frees == f0 + 1);
  // capture after a warm-up on the capturing stream: the same block, nothing allocated
  void* w0 = call(c, 100, 4000);
  capturing.insert(S(100));
  int syncs = device_syncs, ms = memsets;
  void* wc = call(c, 100, 4000);
  CHECK(wc == w0 && device_syncs == syncs && memsets == ms);
  capturing.erase(S(100));
  // many streams later the captured block is still allocated
  for (int s = 200; s < 260; ++s) call(c, s, 1000);
  CHECK(live.count(wc));
  // the captured stream grows: the old block is retained, a new one allocated
  void* wbig = call(c, 100, 100000);
  CHECK(wbig != wc && live.count(wc) && live.count(wbig) && !c.retained.empty());
  // a capture on a new stream while the cache is full: no device synchronisation during it
  for (int s = 300; freeable(c) < kCap; ++s) call(c, s, 1000);
  capturing.insert(S(400));
  syncs = device_syncs;
  void* wn = call(c, 400, 5000);
  // growth during the capture: no stream synchronisation, the first block kept
  void* wn2 = call(c, 400, 50000);
  CHECK(device_syncs == syncs && wn2 != wn && live.count(wn) && live.count(wn2));
  capturing.erase(S(400));
  for (int s = 500; s < 560; ++s) call(c, s, 1000);
  for (void* p : graph_refs) CHECK(live.count(p));
  std::printf("ok: %zu live blocks, %zu entries (%zu freeable), %zu retained, %d device syncs\n", live.size(),
              c.live.size(), freeable(c), c.retained.size(), device_syncs);
  return 0;
}
