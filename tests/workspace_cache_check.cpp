// Host-only check of the per-stream workspace cache policy (workspace_cache.h) on fake CUDA
// calls. The fakes assert the safety rules: no block that a captured graph refers to is ever
// freed; a block is freed on another stream only after that stream waited for the block's last
// use; nothing is freed while the requesting stream is being captured; and a call on a stream
// whose reserved workspace fits allocates, frees and records nothing. Nothing in the policy can
// synchronise: the fake API has no synchronisation call at all.
// Prints "ok" and exits 0 when every scenario holds.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <set>

#include "workspace_cache.h"

namespace {

struct FakeStream;
using Stream = FakeStream*;
struct FakeEvent;
using Event = FakeEvent*;

std::map<void*, Stream> live;             // block -> stream it was last used on (allocation stream at first)
std::set<void*> graph_refs;               // blocks a captured launch refers to
std::set<Stream> capturing;
std::map<Event, Stream> recorded;         // event -> stream it was last recorded on
std::map<Stream, std::set<Stream>> waited;   // stream -> streams whose recorded point it waited for
int mallocs = 0, frees = 0, memsets = 0, records = 0, events = 0;

#define CHECK(cond)                                                            \
  do {                                                                         \
    if (!(cond)) {                                                             \
      std::fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
      std::exit(1);                                                            \
    }                                                                          \
  } while (0)

struct FakeApi {
  using Stream = ::Stream;
  using Event = ::Event;
  static int is_capturing(Stream s, bool* c) {
    *c = capturing.count(s) != 0;
    return 0;
  }
  static int malloc(void** p, size_t n) {
    *p = std::malloc(n);
    live[*p] = nullptr;
    ++mallocs;
    return 0;
  }
  static int malloc_async(void** p, size_t n, Stream s) {
    CHECK(!capturing.count(s));
    *p = std::malloc(n);
    live[*p] = s;
    ++mallocs;
    return 0;
  }
  static int free_async(void* p, Stream s) {
    CHECK(!capturing.count(s));
    CHECK(live.count(p));
    CHECK(!graph_refs.count(p));
    const Stream user = live[p];
    CHECK(user == s || waited[s].count(user));   // ordered after its last use
    live.erase(p);
    std::free(p);
    ++frees;
    return 0;
  }
  static int memset_async(void*, size_t, Stream) {
    ++memsets;
    return 0;
  }
  static int event_create(Event* e) {
    *e = reinterpret_cast<Event>(static_cast<uintptr_t>(0x100000 + 16 * (++events)));
    return 0;
  }
  static int event_destroy(Event e) {
    recorded.erase(e);
    return 0;
  }
  static int event_record(Event e, Stream s) {
    CHECK(!capturing.count(s));
    recorded[e] = s;
    ++records;
    return 0;
  }
  static int stream_wait_event(Stream s, Event e) {
    CHECK(recorded.count(e));
    waited[s].insert(recorded[e]);
    return 0;
  }
};

constexpr size_t kCap = 16;
using Cache = dg::WorkspaceCache<Stream, Event>;

Stream S(int i) { return reinterpret_cast<Stream>(static_cast<uintptr_t>(0x1000 + 16 * i)); }

// One GEMM call on stream s needing `bytes`: acquire, "launch" (the block is used on s), release.
void* call(Cache& c, int s, size_t bytes) {
  void* p = nullptr;
  size_t idx = 0;
  CHECK((dg::acquire<FakeApi, kCap>(c, S(s), bytes, &p, &idx) == 0));
  CHECK(p && live.count(p));
  live[p] = S(s);
  if (capturing.count(S(s))) graph_refs.insert(p);   // the captured launch refers to it
  CHECK((dg::release<FakeApi>(c, idx, S(s)) == 0));
  return p;
}

size_t freeable(const Cache& c) {
  size_t n = 0;
  for (const auto& w : c.live) n += !w.captured && !w.reserved;
  return n;
}

}  // namespace

int main() {
  Cache c;
  // streams come and go: at most kCap freeable entries, each eviction ordered after the last use
  for (int r = 0; r < 3; ++r)
    for (int s = 0; s < 40; ++s) {
      call(c, s, 1000);
      CHECK(freeable(c) <= kCap);
    }
  CHECK(frees > 0 && live.size() <= kCap);
  // the same stream reuses its block; a larger request frees the old one in its own order
  void* u0 = call(c, 600, 100);
  CHECK(call(c, 600, 100) == u0);
  const int f0 = frees;
  void* u1 = call(c, 600, 10000);
  CHECK(u1 != u0 && !live.count(u0) && frees == f0 + 1);
  // a reserved workspace: calls that fit it allocate, free, zero and record nothing
  CHECK((dg::reserve<FakeApi, kCap>(c, S(700), 1 << 20) == 0));
  CHECK(dg::workspace_bytes(c, S(700)) == size_t(1) << 20);
  int m0 = mallocs, fr0 = frees, ms0 = memsets, rec0 = records;
  void* r0 = call(c, 700, 4096);
  for (int i = 0; i < 10; ++i) CHECK(call(c, 700, 1 << 20) == r0);
  CHECK(mallocs == m0 && frees == fr0 && memsets == ms0 && records == rec0);
  // it survives any number of other streams (never evicted)
  for (int s = 800; s < 900; ++s) call(c, s, 1000);
  CHECK(live.count(r0) && freeable(c) <= kCap);
  // a call needing more than was reserved grows it, in stream order
  void* r1 = call(c, 700, 2 << 20);
  CHECK(r1 != r0 && !live.count(r0) && dg::workspace_bytes(c, S(700)) >= size_t(2) << 20);
  // reserve with 0 bytes pins what a stream already has
  void* p9 = call(c, 900, 5000);
  CHECK((dg::reserve<FakeApi, kCap>(c, S(900), 0) == 0));
  for (int s = 1000; s < 1100; ++s) call(c, s, 1000);
  CHECK(live.count(p9));
  // release frees it in its stream's order
  CHECK((dg::reserve_release<FakeApi>(c, S(900)) == 0));
  CHECK(!live.count(p9) && dg::workspace_bytes(c, S(900)) == 0);
  // capture after a warm-up on the capturing stream: the same block, nothing allocated
  void* w0 = call(c, 100, 4000);
  capturing.insert(S(100));
  m0 = mallocs;
  ms0 = memsets;
  void* wc = call(c, 100, 4000);
  CHECK(wc == w0 && mallocs == m0 && memsets == ms0);
  CHECK((dg::reserve<FakeApi, kCap>(c, S(100), 1 << 20) == -1));   // refused during a capture
  CHECK((dg::reserve_release<FakeApi>(c, S(100)) == -1));
  capturing.erase(S(100));
  // many streams later the captured block is still allocated
  for (int s = 200; s < 260; ++s) call(c, s, 1000);
  CHECK(live.count(wc));
  // the captured stream grows: the old block is retained, a new one allocated
  void* wbig = call(c, 100, 100000);
  CHECK(wbig != wc && live.count(wc) && live.count(wbig) && !c.retained.empty());
  // releasing a stream whose workspace a graph refers to keeps the block
  capturing.insert(S(150));
  void* g150 = call(c, 150, 3000);
  capturing.erase(S(150));
  CHECK((dg::reserve_release<FakeApi>(c, S(150)) == 0) && live.count(g150));
  // a capture on a new stream while the cache is full: nothing freed or evicted during it
  for (int s = 300; freeable(c) < kCap; ++s) call(c, s, 1000);
  capturing.insert(S(400));
  const int f1 = frees;
  void* wn = call(c, 400, 5000);
  // growth during the capture: the first block kept
  void* wn2 = call(c, 400, 50000);
  CHECK(frees == f1 && wn2 != wn && live.count(wn) && live.count(wn2));
  capturing.erase(S(400));
  for (int s = 500; s < 560; ++s) call(c, s, 1000);
  for (void* p : graph_refs) CHECK(live.count(p));
  std::printf("ok: %zu live blocks, %zu entries (%zu freeable), %zu retained, %d frees, %d mallocs\n", live.size(),
              c.live.size(), freeable(c), c.retained.size(), frees, mallocs);
  return 0;
}
