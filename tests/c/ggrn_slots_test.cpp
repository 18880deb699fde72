// Host test of the claim-word ownership rule (gated_group_rmsnorm_gb300/csrc/
// ggrn_slots.h): the tests build it with the host C++ compiler and run it.
// Each scenario plays launches on streams against a table of slots, with the
// completion of each slot's last launch under the test's control, and checks
// that no slot is ever given to a launch while another stream's launch on it
// is still running.
#include <cstdio>
#include <cstdlib>

#include "ggrn_slots.h"

using ggrn::ClaimSlot;
using ggrn::pick_claim_slot;

namespace {

constexpr int N = 4;
ClaimSlot slots[N];
bool running[N];  // the slot's last launch has not completed
int failures = 0;

void expect(bool ok, const char* what) {
  if (!ok) {
    std::printf("FAIL %s\n", what);
    ++failures;
  }
}

// One launch on `stream`: pick, check the rule, mark the slot running.
int launch(uintptr_t stream, bool shared_handle, unsigned start) {
  const int i = pick_claim_slot(slots, N, stream, shared_handle, start,
                                [](int k) { return !running[k]; });
  if (i >= 0) {
    const bool same_stream = slots[i].used && slots[i].owner == stream && !shared_handle;
    expect(!running[i] || same_stream, "slot given while another stream's launch runs");
    slots[i].owner = stream;
    slots[i].used = true;
    running[i] = true;
  }
  return i;
}

void reset() {
  for (int i = 0; i < N; ++i) slots[i] = ClaimSlot(), running[i] = false;
}

}  // namespace

int main() {
  const uintptr_t A = 0x1000, B = 0x2000, C = 0x3000, PT = 0x2;
  // one stream keeps its slot, launch after launch, running or not
  reset();
  const int a0 = launch(A, false, 0);
  expect(a0 == 0, "first launch takes slot 0");
  expect(launch(A, false, 1) == a0, "same stream reuses its running slot");
  // another stream never gets a slot whose launch is still running
  const int b0 = launch(B, false, 0);
  expect(b0 >= 0 && b0 != a0, "second stream takes another slot");
  // a completed launch frees its slot for another stream
  running[a0] = false;
  const int c0 = launch(C, false, static_cast<unsigned>(a0));
  expect(c0 == a0, "completed slot passes to a third stream");
  // A's slot is gone: A takes a free one, not C's running slot
  const int a1 = launch(A, false, 0);
  expect(a1 != c0 && a1 != b0 && a1 >= 0, "stream whose slot was taken picks a free one");
  // every slot running on other streams: no slot (static schedule)
  reset();
  for (int i = 0; i < N; ++i) launch(0x100 + i, false, static_cast<unsigned>(i));
  expect(launch(B, false, 0) == -1, "all slots busy: static schedule");
  // the per-thread default stream handle is shared by many streams: it never
  // reuses a running slot, even one it used itself
  reset();
  const int p0 = launch(PT, true, 0);
  expect(p0 == 0, "per-thread stream takes a free slot");
  const int p1 = launch(PT, true, 0);
  expect(p1 != p0, "per-thread stream does not reuse a running slot");
  running[p0] = false;
  expect(launch(PT, true, 0) == p0, "per-thread stream reuses a completed slot");
  // many streams at random, the rule checked at every launch
  reset();
  unsigned seed = 12345;
  for (int t = 0; t < 100000; ++t) {
    seed = seed * 1103515245u + 12345u;
    const uintptr_t s = 0x100 + ((seed >> 16) % 6);
    if ((seed >> 8) % 3 == 0) running[(seed >> 4) % N] = false;
    launch(s, s == 0x100, seed % N);
  }
  std::printf("failures %d\n", failures);
  return failures == 0 ? 0 : 1;
}
