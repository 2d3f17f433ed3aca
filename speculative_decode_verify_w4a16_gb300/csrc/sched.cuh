// Work schedule of the linear kernels over the packed (row-tile, group) units.
//
// The U units are cut into R rounds; round r covers the contiguous unit range
// [rb[r], rb[r+1]) and is split evenly into C items (C = the grid size).
// Round sizes shrink geometrically, so the first items are long contiguous
// runs (few split tiles) and the last ones are short (the grid finishes
// together even when some SMs stream faster than others).
//
// CTA c takes items c, c + C, ... in order: the assignment is known before
// the kernel waits for the grid it depends on, so the weight stream can start
// at once. Item boundaries depend only on (U, C, rb), never on timing, and so
// do the partial-sum slots of split tiles (slot = item index) and the order in
// which a tile's partials are added: results are bitwise reproducible.
#pragma once

#include <stdint.h>

namespace w4a16 {

constexpr int kMaxRounds = 8;

struct ItemSched {
  int64_t rb[kMaxRounds + 1];  // round r covers units [rb[r], rb[r + 1]); rb[0] = 0, rb[R] = U
  int32_t R;                   // rounds
  int32_t C;                   // items per round
};

// First unit of item i, for i in [0, R*C]; item_begin(R*C) = U.
__host__ __device__ __forceinline__ int64_t item_begin(const ItemSched& s, int i) {
  const int r = i / s.C;
  if (r >= s.R) return s.rb[s.R];
  const int64_t j = i - r * s.C;
  return s.rb[r] + j * (s.rb[r + 1] - s.rb[r]) / s.C;
}

// Item that holds unit u (every round holds at least C units, so no item is
// empty).
__host__ __device__ __forceinline__ int item_owner(const ItemSched& s, int64_t u) {
  int r = 0;
  while (r + 1 < s.R && u >= s.rb[r + 1]) ++r;
  const int64_t len = s.rb[r + 1] - s.rb[r];
  return r * s.C + (int)(((u - s.rb[r] + 1) * s.C - 1) / len);
}

// Rounds for U units over C items (U >= C): each round takes half of what is
// left until items would drop below min_units, or max_rounds is reached; the
// last round takes the rest.
inline ItemSched make_item_sched(int64_t U, int C, int min_units, int max_rounds) {
  ItemSched s = {};
  s.C = C;
  if (max_rounds < 1) max_rounds = 1;
  if (max_rounds > kMaxRounds) max_rounds = kMaxRounds;
  int64_t start = 0, rem = U;
  int r = 0;
  while (true) {
    s.rb[r] = start;
    if (r == max_rounds - 1 || rem <= 2 * (int64_t)C * min_units) {
      s.rb[r + 1] = U;
      s.R = r + 1;
      break;
    }
    const int64_t len = rem / 2;
    start += len;
    rem -= len;
    ++r;
  }
  return s;
}

// Counter layout at the start of every workspace (int32 indices).
constexpr int kTileCounterBase = 64;  // per (tile, warp) split-tile counters (ints 0..63 reserved)

}  // namespace w4a16
