// Launch slots for the streaming CE kernels: the words a launch shares across its CTAs.
//   rows   a counter of claimed rows (dynamic row claims: a CTA that finishes its rows early
//          takes the next unclaimed one, so no CTA is left with a longer share at the end)
//   done   the count of finished CTAs (the last one reduces the losses)
//   err    the first device error code of the launch
// They live in a device array of the including translation unit, zero whenever no launch holds
// a slot: zero-initialised at module load, and put back to zero by the CTA that finishes last,
// which also writes the caller's status word (the error code, or 0) with a plain store.  So no
// launch needs a separate clearing step before it.  The host hands each launch the next slot
// round-robin; a slot comes round again kLaunchSlots launches of the same kernel later, so at
// most that many of them may be in flight at once (on any streams).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace vce {
namespace slots {

struct alignas(16) LaunchSlot {
    unsigned int rows;
    int done;
    int err;
    int pad;
};
constexpr int kLaunchSlots = 1024;

// one array (and one round-robin counter) per translation unit that includes this header
static __device__ LaunchSlot g_launch_slots[kLaunchSlots];
static std::atomic<unsigned int> g_next_slot{0};

inline int next_slot() { return (int)(g_next_slot.fetch_add(1u, std::memory_order_relaxed) % kLaunchSlots); }

}  // namespace slots
}  // namespace vce
