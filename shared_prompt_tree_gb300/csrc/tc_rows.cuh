// Row geometry of the query-side tensor-core kernels (the forward and the backward's
// query side): where a query row's keys lie in each KV tile of its walk.
//
// AugTree paper, Sec. 3.2 Eq. 1 (the row's valid keys: the whole prompt of its group,
// then its own branch up to itself; causal over the prompt for prefill rows) and Sec. 3.3
// (the prompt-part and own-part states merge associatively; one running state crosses
// both parts).
#pragma once

#include "common.cuh"

namespace augtree {
namespace tc {

// Where the row's keys come from in KV tile j: prompt tiles first, then the own-branch
// tiles, and the valid columns [lo, hi] of the row in that tile.
struct FwdRowGeom {
  int64_t row;      // global query row (prompt or response rows)
  bool row_ok;      // row < end of its query tile's group
  bool prefill;
  int64_t bs;       // first response row of the row's branch (replay rows)
  int64_t p0, p_end;  // the group's prompt keys
  int64_t own0;     // first key of the own-branch tiles
  int n_a;          // number of prompt tiles
  int bn;           // keys per tile
  int j0;           // first KV tile of the item (a split item's chunk; 0 otherwise)
};

// Valid columns of the item's j-th KV tile (tile j0 + j of the row's walk), clamped to
// [-1, 128].  Rows and keys are int32 offsets (the descriptors are int32), so every
// difference below fits in 32 bits; 32-bit arithmetic measured 1.4 % faster in the
// forward than 64-bit.
__device__ __forceinline__ void fwd_valid_cols(const FwdRowGeom& g, int j_local, int& lo_i, int& hi_i) {
  const int j = j_local + g.j0;
  const bool own = j >= g.n_a;
  const int key0 = own ? (int)g.own0 + (j - g.n_a) * g.bn : (int)g.p0 + j * g.bn;
  const int row = (int)g.row;
  int lo = 0, hi;
  if (g.prefill) {
    hi = row - key0;
  } else if (!own) {
    hi = (int)g.p_end - 1 - key0;
  } else {
    lo = (int)g.bs - key0;
    hi = row - key0;
  }
  if (!g.row_ok) {
    lo = 1;
    hi = 0;
  }
  lo_i = min(max(lo, -1), 128);
  hi_i = min(max(hi, -1), 128);
}

}  // namespace tc
}  // namespace augtree
