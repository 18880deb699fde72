// ggrn_slots.h -- which unit-claim word a streaming launch may use.
//
// The streaming kernel's dynamic schedule hands out units from a 64-bit
// claim word in device memory (epoch << 32 | next).  A word must never serve
// two launches that run at the same time: each would keep replacing the
// other's epoch and restarting, which keeps the output correct but need not
// end.  So the host gives a word to one launch at a time:
//
//   * launches on the same stream may share a word: each one's claims come
//     after its programmatic-dependent-launch wait, which returns only once
//     the previous kernel of the stream (and, through it, every earlier one)
//     has completed;
//   * a word last used on another stream is taken only once that stream's
//     launch on it has completed (an event recorded after the launch);
//   * the per-thread default stream has one handle for many streams, so a
//     word it used counts as another stream's;
//   * when no word qualifies the launch takes the static schedule (no word).
//
// This header holds the decision only (no CUDA calls), so that the host
// tests can exercise it with a plain C++ compiler.
#pragma once

#include <stdint.h>

namespace ggrn {

struct ClaimSlot {
  uintptr_t owner = 0;  // stream handle of the slot's last launch
  bool used = false;    // the slot has had a launch
};

// The slot for a launch on `stream`: first a slot this stream used last
// (unless `shared_handle`), else the first of slots start, start+1, ... that
// is unused or whose last launch has completed (done(i)); -1 when none is.
template <class Done>
int pick_claim_slot(const ClaimSlot* slots, int n, uintptr_t stream, bool shared_handle,
                    unsigned start, Done done) {
  if (!shared_handle) {
    for (int i = 0; i < n; ++i)
      if (slots[i].used && slots[i].owner == stream) return i;
  }
  for (int k = 0; k < n; ++k) {
    const int i = static_cast<int>((start + static_cast<unsigned>(k)) % static_cast<unsigned>(n));
    if (!slots[i].used || done(i)) return i;
  }
  return -1;
}

}  // namespace ggrn
